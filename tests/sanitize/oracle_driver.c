/*
 * Runs every oracle routine once on small ragged inputs, compiled together
 * with the oracle source under AddressSanitizer and UndefinedBehaviorSanitizer
 * (tests/test_sanitizers.py).  Test infrastructure: it checks memory safety
 * and undefined behaviour of the oracle, not its values (the pins do that).
 * Exit status 0 and no sanitizer report is a pass.
 */
#include "../../oracle/fp8z1_oracle.c"

#include <stdio.h>

static float frand(uint32_t* s)
{
    *s = *s * 1664525u + 1013904223u;
    return ((float)(*s >> 8) / 16777216.0f - 0.5f) * 2.0f;
}

int main(void)
{
    const orc_shape shapes[] = {{1, 300, 200}, {3, 129, 257}, {1, 1, 1}, {2, 128, 128}, {1, 17, 690}};
    const int32_t n = (int32_t)(sizeof shapes / sizeof shapes[0]);
    const int64_t nblk = oracle_count_blocks(shapes, n);
    const int64_t padded = nblk * ORC_BLOCK_ELEMS;
    uint32_t seed = 12345u;

    orc_block* lut = (orc_block*)malloc(sizeof(orc_block) * (size_t)nblk);
    oracle_build_lut(shapes, n, lut);
    for (int32_t dp = 1; dp <= 5; ++dp)
        for (int32_t r = 0; r < dp; ++r) {
            int64_t b0, b1;
            oracle_shard_range(nblk, dp, r, &b0, &b1);
        }

    /* row-major params of every element size, folded and unfolded back over
       the whole range and a sub-range */
    const int32_t sizes[] = {1, 2, 4};
    for (int si = 0; si < 3; ++si) {
        const int32_t esz = sizes[si];
        void* src[5];
        void* back[5];
        for (int32_t i = 0; i < n; ++i) {
            const size_t bytes = (size_t)(shapes[i].E * shapes[i].R * shapes[i].C) * (size_t)esz;
            src[i] = malloc(bytes);
            back[i] = calloc(1, bytes);
            for (size_t b = 0; b < bytes; ++b) ((uint8_t*)src[i])[b] = (uint8_t)(b * 31u + (size_t)i);
        }
        void* folded = malloc((size_t)padded * (size_t)esz);
        if (oracle_fold(shapes, n, (const void* const*)src, folded, esz, 0, nblk) != 0) return 1;
        if (oracle_unfold(shapes, n, folded, back, esz, 0, nblk) != 0) return 1;
        if (oracle_fold(shapes, n, (const void* const*)src, folded, esz, 2, nblk - 1) != 0) return 1;
        if (oracle_unfold(shapes, n, folded, back, esz, 2, nblk - 1) != 0) return 1;
        free(folded);
        for (int32_t i = 0; i < n; ++i) {
            free(src[i]);
            free(back[i]);
        }
    }

    /* norm, clip, step, quantiser, monitors, scaler */
    float* g = (float*)malloc(sizeof(float) * (size_t)padded);
    float* p = (float*)malloc(sizeof(float) * (size_t)padded);
    float* m = (float*)calloc((size_t)padded, sizeof(float));
    float* v = (float*)calloc((size_t)padded, sizeof(float));
    uint8_t* q = (uint8_t*)malloc((size_t)padded);
    float* scales = (float*)malloc(sizeof(float) * (size_t)nblk);
    for (int64_t i = 0; i < padded; ++i) {
        g[i] = frand(&seed) * 1024.0f;
        p[i] = frand(&seed) * 0.02f;
    }
    g[5] = 1e-40f;   /* subnormal */
    g[6] = 3.0e38f;  /* a square that overflows float */
    orc_sumsq_acc acc, acc2;
    oracle_acc_init(&acc);
    oracle_acc_init(&acc2);
    oracle_acc_add(&acc, g, padded / 2);
    oracle_acc_add(&acc2, g + padded / 2, padded - padded / 2);
    oracle_acc_merge(&acc, &acc2);
    double s = oracle_acc_result(&acc), s2;
    int32_t fi;
    oracle_sumsq(g, padded, &s2, &fi);
    g[6] = 0.5f;
    oracle_sumsq(g, padded, &s, &fi);
    double gn, cc;
    int32_t ap;
    oracle_clip_coef(s, 0.5f, 1024.0f, &gn, &cc, &ap);
    orc_hp hp = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 0.5f, 1024.0f, 1};
    for (int64_t t = 1; t <= 3; ++t) {
        hp.step = t;
        oracle_step(&hp, s, fi, g, p, m, v, q, scales, nblk);
    }
    oracle_step(&hp, s, 1, g, p, m, v, q, scales, nblk); /* skipped */
    for (int64_t k = 0; k < nblk; ++k) {
        double cosv;
        int64_t under;
        oracle_quant_monitor(p + k * ORC_BLOCK_ELEMS, q + k * ORC_BLOCK_ELEMS, scales[k], ORC_BLOCK_ELEMS,
                             &cosv, &under);
    }
    uint8_t codes[256];
    float vals[256];
    for (int c = 0; c < 256; ++c) codes[c] = (uint8_t)c;
    oracle_e4m3_decode_n(codes, vals, 256);
    for (int c = 0; c < 256; ++c)
        if (c != 0x7F && c != 0xFF) (void)oracle_e4m3_encode(vals[c]);
    oracle_e4m3_encode_n(g, q, padded);
    oracle_quantise_block(p, q, scales);
    orc_scaler sc = {65536.0f, 0, 0, 2};
    for (int i = 0; i < 6; ++i) oracle_scaler_update(&sc, i == 3);

    /* the param-wise split */
    int32_t owner[5];
    int64_t bucket[8];
    for (int32_t dp = 1; dp <= 8; ++dp) oracle_paramwise_split(shapes, n, dp, owner, bucket);

    /* MXFP8: groups of 32 */
    const int64_t ng = padded / ORC_MX_GROUP;
    uint8_t* e8 = (uint8_t*)malloc((size_t)ng);
    oracle_mx_quantise_group(p, q, e8);
    for (int c = 0; c < 256; ++c) (void)oracle_e8m0_decode((uint8_t)c);
    memset(m, 0, sizeof(float) * (size_t)padded);
    memset(v, 0, sizeof(float) * (size_t)padded);
    oracle_mx_step(&hp, s, 0, g, p, m, v, q, e8, ng);

    free(e8);
    free(g);
    free(p);
    free(m);
    free(v);
    free(q);
    free(scales);
    free(lut);
    printf("oracle driver ok\n");
    return 0;
}
