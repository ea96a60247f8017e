/*
 * fp8z1 oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what the blockwise-FP8
 * ZeRO-1 optimizer step computes.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  It shares
 * no code, header, table or helper with the CUDA library: every definition
 * below is written out again from the pages.
 *
 * Sources (page title, section):
 *   [ZF] "面向 Blockwise FP8 量化的 ZeRO 优化器设计" (A ZeRO Optimizer Design
 *        for Blockwise FP8 Quantization):
 *        - §Blockwise 量化: one scale per 128x128 sub-matrix of a weight.
 *        - §块粒度切分 (block-wise split): pad the quantised dims to multiples
 *          of 128, record real and padded sizes, shard on block edges.
 *        - §参数布局变换 (layout transform): the fold / unfold view-permute
 *          pseudocode; fold makes each 128x128 block contiguous.
 *        - §总结 (modified update flow): fold grads, slice, elementwise update,
 *          quantise FP8 + scales from the FP32 master, unfold.
 *   [DS] "DeepSpeed ZeRO 优化":
 *        - §三 Stage 1/2 step order: global norm -> loss-scale update ->
 *          unscale+clip -> optimizer step -> low-precision copy.
 *        - §六 Loss Scaling: on inf/nan halve S and skip; grow after N clean steps.
 *        - §七 梯度裁剪: global = scaled_global / loss_scale;
 *          clip_coef = max_norm / (global + 1e-6); multiply when clip_coef < 1.
 *   [FP8] "FP8训练技术与万亿参数模型优化实践" §1.1: the FP8 format is E4M3.
 *   E4M3 bit layout: OCP 8-bit floating point specification (OFP8), E4M3
 *   ("FN": bias 7, no infinities, S.1111.111 is NaN, max normal 448).
 *
 * Readings where the pages are silent:
 *   - AdamW: decoupled weight decay, bias correction, eps added after the
 *     square root of the bias-corrected second moment, t starting at 1.
 *     Arithmetic in FP32 (the pages keep master params, grads and moments in
 *     FP32), in the one operation order written out in adamw_element().
 *   - block scale = amax / 448 (1.0 when amax == 0); code = E4M3 of p / scale,
 *     round-to-nearest-even, finite overflow saturates to +-448, sign kept.
 *   - grad norm: the exact sum of squares of the stored FP32 grads, rounded
 *     once to double; then the clip scalars in double; the clip factor is
 *     applied to the FP32 grads as an FP32 number.
 *   - shard size for DP size D: ceil(nblk / D) blocks, last rank shorter.
 *
 * Pins (tests/): PyTorch CPU view/permute for fold, math.fsum for the exact
 * norm, torch.optim.AdamW and closed-form trajectories for the update,
 * torch.float8_e4m3fn and brute-force nearest search for E4M3.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off (no contraction of a*b+c; the only
 * fused multiply-adds are the explicit fmaf calls).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_TILE 128
#define ORC_BLOCK_ELEMS (ORC_TILE * ORC_TILE)

typedef struct {
    int64_t E, R, C; /* 2-D weights use E = 1 */
} orc_shape;

/* One entry of the block lookup table: flat block index -> where it lives. */
typedef struct {
    int64_t param;     /* index into the shape list */
    int64_t expert;    /* e in [0, E) */
    int64_t row_block; /* rb in [0, ceil(R/128)) */
    int64_t col_block; /* cb in [0, ceil(C/128)) */
    int64_t rows_real; /* min(128, R - 128*rb) */
    int64_t cols_real; /* min(128, C - 128*cb) */
} orc_block;

typedef struct {
    float lr, beta1, beta2, eps, weight_decay, max_norm, loss_scale;
    int64_t step; /* t >= 1 */
} orc_hp;

/* ========================================================================= */
/* Layout [ZF §块粒度切分, §参数布局变换]                                     */
/* ========================================================================= */

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Blocks of one param: E * (R padded to 128)/128 * (C padded to 128)/128. */
int64_t oracle_param_blocks(const orc_shape* s)
{
    return s->E * ceil_div(s->R, ORC_TILE) * ceil_div(s->C, ORC_TILE);
}

int64_t oracle_count_blocks(const orc_shape* shapes, int32_t n)
{
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i) total += oracle_param_blocks(&shapes[i]);
    return total;
}

/* Params in the given order; inside a param the blocks follow the order that
 * view(E, R/128, 128, C/128, 128).permute(0, 1, 3, 2, 4).view(-1, 128, 128)
 * produces: expert e, then row block, then column block. */
void oracle_build_lut(const orc_shape* shapes, int32_t n, orc_block* lut)
{
    int64_t k = 0;
    for (int32_t i = 0; i < n; ++i) {
        int64_t rbs = ceil_div(shapes[i].R, ORC_TILE);
        int64_t cbs = ceil_div(shapes[i].C, ORC_TILE);
        for (int64_t e = 0; e < shapes[i].E; ++e)
            for (int64_t rb = 0; rb < rbs; ++rb)
                for (int64_t cb = 0; cb < cbs; ++cb) {
                    orc_block b;
                    b.param = i;
                    b.expert = e;
                    b.row_block = rb;
                    b.col_block = cb;
                    b.rows_real = shapes[i].R - ORC_TILE * rb;
                    if (b.rows_real > ORC_TILE) b.rows_real = ORC_TILE;
                    b.cols_real = shapes[i].C - ORC_TILE * cb;
                    if (b.cols_real > ORC_TILE) b.cols_real = ORC_TILE;
                    lut[k++] = b;
                }
    }
}

/* Uniform split of the block list over D ranks, cut on block edges. */
void oracle_shard_range(int64_t nblk, int32_t dp, int32_t rank, int64_t* b0, int64_t* b1)
{
    int64_t per = ceil_div(nblk, dp);
    int64_t lo = per * rank;
    int64_t hi = per * (rank + 1);
    if (lo > nblk) lo = nblk;
    if (hi > nblk) hi = nblk;
    *b0 = lo;
    *b1 = hi;
}

/* Byte offset of element (e, row, col) of a row-major [E, R, C] tensor. */
static int64_t rowmajor_offset(const orc_shape* s, int64_t e, int64_t row, int64_t col, int32_t esz)
{
    return ((e * s->R + row) * s->C + col) * esz;
}

/* fold over the blocks [b0, b1): for block k and (r, c) in 128 x 128,
 *   dst[(k - b0) * 16384 + r * 128 + c] = src_param[e][128 rb + r][128 cb + c]
 * when the element is real, and 0 when it is padding.  esz = 1, 2 or 4 bytes;
 * the copy is bitwise.  Returns 0, or -1 when the LUT cannot be allocated. */
int oracle_fold(const orc_shape* shapes, int32_t n, const void* const* src, void* dst,
                int32_t esz, int64_t b0, int64_t b1)
{
    int64_t nblk = oracle_count_blocks(shapes, n);
    orc_block* lut = (orc_block*)malloc(sizeof(orc_block) * (size_t)(nblk ? nblk : 1));
    if (!lut) return -1;
    oracle_build_lut(shapes, n, lut);
    uint8_t* out = (uint8_t*)dst;
    for (int64_t k = b0; k < b1; ++k) {
        const orc_block* b = &lut[k];
        const orc_shape* s = &shapes[b->param];
        const uint8_t* in = (const uint8_t*)src[b->param];
        for (int64_t r = 0; r < ORC_TILE; ++r)
            for (int64_t c = 0; c < ORC_TILE; ++c) {
                uint8_t* d = out + ((k - b0) * ORC_BLOCK_ELEMS + r * ORC_TILE + c) * esz;
                if (r < b->rows_real && c < b->cols_real)
                    memcpy(d, in + rowmajor_offset(s, b->expert, ORC_TILE * b->row_block + r,
                                                   ORC_TILE * b->col_block + c, esz),
                           (size_t)esz);
                else
                    memset(d, 0, (size_t)esz);
            }
    }
    free(lut);
    return 0;
}

/* unfold over the blocks [b0, b1): the inverse of fold on the real elements;
 * the padding of the block buffer is dropped and nothing else is written. */
int oracle_unfold(const orc_shape* shapes, int32_t n, const void* src, void* const* dst,
                  int32_t esz, int64_t b0, int64_t b1)
{
    int64_t nblk = oracle_count_blocks(shapes, n);
    orc_block* lut = (orc_block*)malloc(sizeof(orc_block) * (size_t)(nblk ? nblk : 1));
    if (!lut) return -1;
    oracle_build_lut(shapes, n, lut);
    const uint8_t* in = (const uint8_t*)src;
    for (int64_t k = b0; k < b1; ++k) {
        const orc_block* b = &lut[k];
        const orc_shape* s = &shapes[b->param];
        uint8_t* out = (uint8_t*)dst[b->param];
        for (int64_t r = 0; r < b->rows_real; ++r)
            for (int64_t c = 0; c < b->cols_real; ++c)
                memcpy(out + rowmajor_offset(s, b->expert, ORC_TILE * b->row_block + r,
                                             ORC_TILE * b->col_block + c, esz),
                       in + ((k - b0) * ORC_BLOCK_ELEMS + r * ORC_TILE + c) * esz, (size_t)esz);
    }
    free(lut);
    return 0;
}

/* ========================================================================= */
/* Global grad norm [DS §七, §六]                                             */
/* ========================================================================= */

/* The sum of squares is accumulated EXACTLY in a fixed-point big integer:
 * a finite float is m * 2^x with m < 2^24 and x in [-149, 104], so its square
 * is m^2 * 2^(2x) with m^2 < 2^48.  Bit i of the accumulator weighs 2^(i-298).
 * Ten 64-bit limbs give 640 bits: 554 for the largest square and 86 of
 * headroom for the count of terms. */
#define ORC_ACC_LIMBS 10
#define ORC_ACC_BIAS 298

typedef struct {
    uint64_t limb[ORC_ACC_LIMBS];
    int32_t found_inf; /* any inf or nan seen */
    int32_t found_nan; /* any nan seen */
} orc_sumsq_acc;

void oracle_acc_init(orc_sumsq_acc* a) { memset(a, 0, sizeof(*a)); }

static void acc_add_square(orc_sumsq_acc* a, float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint32_t ef = (bits >> 23) & 0xFFu;
    uint64_t mant = bits & 0x7FFFFFu;
    if (ef == 0xFFu) { /* inf or nan */
        a->found_inf = 1;
        if (mant) a->found_nan = 1;
        return;
    }
    int32_t x2;
    if (ef == 0) {
        x2 = -149; /* subnormal: 0.mant * 2^-126 = mant * 2^-149 */
    } else {
        mant |= 0x800000u;
        x2 = (int32_t)ef - 150;
    }
    if (mant == 0) return;
    uint64_t sq = mant * mant; /* < 2^48 */
    int32_t shift = 2 * x2 + ORC_ACC_BIAS; /* in [0, 506] */
    int32_t li = shift / 64, off = shift % 64;
    uint64_t lo = sq << off;
    uint64_t hi = off ? (sq >> (64 - off)) : 0;
    uint64_t old = a->limb[li];
    a->limb[li] = old + lo;
    uint64_t carry = a->limb[li] < old;
    uint64_t add = hi + carry;
    for (int32_t j = li + 1; add && j < ORC_ACC_LIMBS; ++j) {
        old = a->limb[j];
        a->limb[j] = old + add;
        add = a->limb[j] < old;
    }
}

void oracle_acc_add(orc_sumsq_acc* a, const float* g, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) acc_add_square(a, g[i]);
}

/* a += b, exactly (big-integer addition of the limbs; flags OR-ed): the sum
 * of two exact partial sums is the exact sum of their terms. */
void oracle_acc_merge(orc_sumsq_acc* a, const orc_sumsq_acc* b)
{
    uint64_t carry = 0;
    for (int32_t j = 0; j < ORC_ACC_LIMBS; ++j) {
        uint64_t s = a->limb[j] + b->limb[j];
        uint64_t c1 = s < a->limb[j];
        uint64_t t = s + carry;
        uint64_t c2 = t < s;
        a->limb[j] = t;
        carry = c1 | c2;
    }
    a->found_inf |= b->found_inf;
    a->found_nan |= b->found_nan;
}

static int acc_bit(const orc_sumsq_acc* a, int64_t i)
{
    return (int)((a->limb[i / 64] >> (i % 64)) & 1u);
}

/* The exact sum rounded once to the nearest double (ties to even).  With an
 * inf or nan among the terms the sum is +inf (nan when a nan was seen). */
double oracle_acc_result(const orc_sumsq_acc* a)
{
    if (a->found_nan) return NAN;
    if (a->found_inf) return INFINITY;
    int64_t top = -1; /* index of the highest set bit */
    for (int64_t i = 64 * ORC_ACC_LIMBS - 1; i >= 0; --i)
        if (acc_bit(a, i)) { top = i; break; }
    if (top < 0) return 0.0;
    int64_t len = top + 1;
    if (len <= 53) { /* exact: fits in limb 0 */
        return ldexp((double)a->limb[0], -ORC_ACC_BIAS);
    }
    uint64_t m = 0; /* the top 53 bits */
    for (int64_t i = top; i >= len - 53; --i) m = (m << 1) | (uint64_t)acc_bit(a, i);
    int round = acc_bit(a, len - 54);
    int sticky = 0;
    for (int64_t i = len - 55; i >= 0 && !sticky; --i) sticky = acc_bit(a, i);
    if (round && (sticky || (m & 1u))) m += 1; /* 2^53 is still exact */
    return ldexp((double)m, (int)(len - 53) - ORC_ACC_BIAS);
}

/* sum of g[i]^2 over n stored (loss-scaled) grads, and the inf/nan flag. */
void oracle_sumsq(const float* g, int64_t n, double* sumsq, int32_t* found_inf)
{
    orc_sumsq_acc a;
    oracle_acc_init(&a);
    oracle_acc_add(&a, g, n);
    *sumsq = oracle_acc_result(&a);
    *found_inf = a.found_inf;
}

/* [DS §七] from the global sum of squares of the loss-scaled grads:
 *   scaled_global_norm = sqrt(sumsq); global_norm = scaled / loss_scale;
 *   clip_coef = max_norm / (global_norm + 1e-6); applied when clip_coef < 1.
 * All in double. */
void oracle_clip_coef(double sumsq, float max_norm, float loss_scale, double* global_norm,
                      double* clip_coef, int32_t* clip_applies)
{
    double scaled = sqrt(sumsq);
    double global = scaled / (double)loss_scale;
    double coef = (double)max_norm / (global + 1e-6);
    *global_norm = global;
    *clip_coef = coef;
    *clip_applies = coef < 1.0;
}

/* ========================================================================= */
/* E4M3 (OCP OFP8 E4M3, the "FN" variant)                                    */
/* ========================================================================= */

/* value of a code: S.EEEE.MMM, bias 7; E = 0 is subnormal (M/8 * 2^-6);
 * S.1111.111 is NaN; there are no infinities. */
float oracle_e4m3_decode(uint8_t q)
{
    int s = q >> 7, E = (q >> 3) & 0xF, M = q & 7;
    float mag;
    if (E == 15 && M == 7)
        mag = NAN;
    else if (E == 0)
        mag = ldexpf((float)M, -9);
    else
        mag = ldexpf((float)(8 + M), E - 10); /* (1 + M/8) * 2^(E-7) */
    return s ? -mag : mag;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating finite overflow to the
 * largest finite value 448 (codes 0x7E / 0xFE); the sign is kept, so -0 and
 * negatives that round to zero give 0x80.  In the binade [2^e, 2^(e+1)) the
 * grid step is 2^(e-3); below 2^-6 the subnormal step 2^-9 continues the
 * e = -6 grid.  Because codes grow monotonically with magnitude, the code is
 * (e + 7) * 8 + n - 8 where n is the rounded multiple of the step; n = 16
 * carries into the next binade by itself. */
uint8_t oracle_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    float a = fabsf(x);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
    int k = 0;
    (void)frexpf(a, &k); /* a = f * 2^k, f in [0.5, 1); a = 0 gives k = 0 */
    int e = (a == 0.0f) ? -6 : k - 1;
    if (e < -6) e = -6;
    float n = nearbyintf(ldexpf(a, 3 - e)); /* default rounding mode: to nearest even */
    int code = (e + 7) * 8 + (int)n - 8;
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)(sign | code);
}

/* ========================================================================= */
/* Fused step [ZF §总结; DS §三, §七]                                         */
/* ========================================================================= */

/* Scalars of one step, derived on the host in double from the FP32
 * hyper-parameters, then rounded to FP32. */
typedef struct {
    float omb1, omb2;     /* 1 - beta1, 1 - beta2 */
    float step_size;      /* lr / (1 - beta1^t) */
    float inv_sqrt_bc2;   /* 1 / sqrt(1 - beta2^t) */
    float decay;          /* 1 - lr * weight_decay */
    float clip;           /* clip_coef as FP32 (used when clip_applies) */
    int32_t clip_applies; /* clip_coef < 1 */
} orc_derived;

static orc_derived derive(const orc_hp* hp, double sumsq)
{
    orc_derived d;
    double t = (double)hp->step;
    double bc1 = 1.0 - pow((double)hp->beta1, t);
    double bc2 = 1.0 - pow((double)hp->beta2, t);
    d.omb1 = (float)(1.0 - (double)hp->beta1);
    d.omb2 = (float)(1.0 - (double)hp->beta2);
    d.step_size = (float)((double)hp->lr / bc1);
    d.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    d.decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    double global, coef;
    oracle_clip_coef(sumsq, hp->max_norm, hp->loss_scale, &global, &coef, &d.clip_applies);
    d.clip = (float)coef;
    return d;
}

/* AdamW on one element, FP32:
 *   g  = g_s / S, then g = g * clip when clip_coef < 1      (unscale, clip)
 *   m  = beta1 m + (1 - beta1) g                            (first moment)
 *   v  = beta2 v + (1 - beta2) g^2                          (second moment)
 *   p  = p (1 - lr wd) - lr * mhat / (sqrt(vhat) + eps),    mhat = m / bc1,
 *        vhat = v / bc2, written as
 *        p (1 - lr wd) - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps). */
static void adamw_element(const orc_hp* hp, const orc_derived* d, float g_s, float* p, float* m,
                          float* v)
{
    float g = g_s / hp->loss_scale;
    if (d->clip_applies) g = g * d->clip;
    float mn = fmaf(hp->beta1, *m, d->omb1 * g);
    float vn = fmaf(hp->beta2, *v, (d->omb2 * g) * g);
    float den = fmaf(sqrtf(vn), d->inv_sqrt_bc2, hp->eps);
    float pn = fmaf(-d->step_size, mn / den, *p * d->decay);
    *m = mn;
    *v = vn;
    *p = pn;
}

/* One block: scale = amax / 448 (1 when amax == 0), codes = E4M3(p / scale). */
void oracle_quantise_block(const float* p, uint8_t* codes, float* scale)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < ORC_BLOCK_ELEMS; ++i) {
        float a = fabsf(p[i]);
        if (a > amax) amax = a;
    }
    float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    for (int64_t i = 0; i < ORC_BLOCK_ELEMS; ++i) codes[i] = oracle_e4m3_encode(p[i] / s);
    *scale = s;
}

/* The optimizer step on nblocks consecutive folded blocks of one shard.
 * sumsq / found_inf are the GLOBAL sum of squares and inf flag.  With
 * found_inf set nothing is written (the step is skipped) and 1 is returned;
 * otherwise master/m/v are updated in place, codes/scales written, 0 returned. */
int oracle_step(const orc_hp* hp, double sumsq, int32_t found_inf, const float* grad,
                float* master, float* m, float* v, uint8_t* codes, float* scales,
                int64_t nblocks)
{
    if (found_inf) return 1;
    orc_derived d = derive(hp, sumsq);
    for (int64_t k = 0; k < nblocks; ++k) {
        int64_t base = k * ORC_BLOCK_ELEMS;
        for (int64_t i = 0; i < ORC_BLOCK_ELEMS; ++i)
            adamw_element(hp, &d, grad[base + i], &master[base + i], &m[base + i], &v[base + i]);
        oracle_quantise_block(master + base, codes + base, &scales[k]);
    }
    return 0;
}

/* ========================================================================= */
/* Dynamic loss scaling and the skip rule [DS §六, §九 Q6]                   */
/* ========================================================================= */

typedef struct {
    float scale;             /* S */
    int64_t step;            /* completed (not skipped) steps t */
    int32_t good_steps;      /* clean steps since the last change of S */
    int32_t growth_interval; /* N */
} orc_scaler;

/* After a step: an inf/nan halves S and the step does not count; otherwise t
 * advances and after N clean steps in a row S doubles. */
void oracle_scaler_update(orc_scaler* s, int32_t found_inf)
{
    if (found_inf) {
        s->scale = s->scale * 0.5f;
        s->good_steps = 0;
        return;
    }
    s->step += 1;
    s->good_steps += 1;
    if (s->good_steps >= s->growth_interval) {
        s->scale = s->scale * 2.0f;
        s->good_steps = 0;
    }
}

/* ========================================================================= */
/* Array forms of the codec, for the tests                                   */
/* ========================================================================= */

void oracle_e4m3_encode_n(const float* x, uint8_t* q, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_n(const uint8_t* q, float* x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) x[i] = oracle_e4m3_decode(q[i]);
}

/* ========================================================================= */
/* Param-wise split [ZF §参数粒度切分]                                        */
/* ========================================================================= */

/* The page's alternative to the block-wise split: sort the FP8 params by size
 * (largest first; equal sizes keep their given order), hand each in turn to
 * the DP bucket holding the fewest elements so far (the lowest bucket index on
 * a tie), then pad every bucket up to the largest one.  Size = E * R * C real
 * elements.  owner[i] = bucket of param i; bucket[b] = elements in bucket b
 * before padding. */
void oracle_paramwise_split(const orc_shape* shapes, int32_t n, int32_t dp, int32_t* owner,
                            int64_t* bucket)
{
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    for (int32_t i = 0; i < n; ++i) order[i] = i;
    /* insertion sort: larger first, ties in index order (stable) */
    for (int32_t i = 1; i < n; ++i) {
        int32_t cur = order[i];
        int64_t sz = shapes[cur].E * shapes[cur].R * shapes[cur].C;
        int32_t j = i - 1;
        while (j >= 0) {
            int32_t o = order[j];
            int64_t so = shapes[o].E * shapes[o].R * shapes[o].C;
            if (so >= sz) break;
            order[j + 1] = o;
            --j;
        }
        order[j + 1] = cur;
    }
    for (int32_t b = 0; b < dp; ++b) bucket[b] = 0;
    for (int32_t t = 0; t < n; ++t) {
        int32_t i = order[t];
        int32_t best = 0;
        for (int32_t b = 1; b < dp; ++b)
            if (bucket[b] < bucket[best]) best = b;
        owner[i] = best;
        bucket[best] += shapes[i].E * shapes[i].R * shapes[i].C;
    }
    free(order);
}

/* ========================================================================= */
/* Quantisation-error monitors ["FP8训练技术与万亿参数模型优化实践" §1.2]         */
/* ========================================================================= */

/* The page watches two numbers: Underflow = zeros / total (healthy below 0.5%)
 * and Distortion = cosine(original, dequantised) (healthy above 0.995).
 * Reading, per block of n values: underflow = the count of non-zero master
 * values whose code decodes to 0 (the host divides by the block's real
 * elements); cosine = sum(p d) / sqrt(sum(p^2) sum(d^2)) with
 * d = decode(q) * scale, in double; 1 when both vectors are 0, 0 when only one
 * is. */
void oracle_quant_monitor(const float* p, const uint8_t* q, float scale, int64_t n, double* cosine,
                          int64_t* underflow)
{
    double pd = 0.0, pp = 0.0, dd = 0.0;
    int64_t under = 0;
    for (int64_t i = 0; i < n; ++i) {
        double dq = (double)oracle_e4m3_decode(q[i]);
        double d = dq * (double)scale;
        double x = (double)p[i];
        pd += x * d;
        pp += x * x;
        dd += d * d;
        if (p[i] != 0.0f && dq == 0.0) ++under;
    }
    if (pp == 0.0 && dd == 0.0)
        *cosine = 1.0;
    else if (pp == 0.0 || dd == 0.0)
        *cosine = 0.0;
    else
        *cosine = pd / sqrt(pp * dd);
    *underflow = under;
}

/* ========================================================================= */
/* MXFP8 [ZF §Blockwise 量化: MXFP8 gives each memory-contiguous block an      */
/* E8M0 scale]; format per the OCP Microscaling (MX) specification v1.0       */
/* ========================================================================= */

#define ORC_MX_GROUP 32

/* E8M0: an unsigned exponent, value 2^(e - 127) for e in [0, 254]; 255 is NaN. */
float oracle_e8m0_decode(uint8_t e)
{
    if (e == 255) return NAN;
    return ldexpf(1.0f, (int)e - 127);
}

/* One group of 32 consecutive values: the shared scale is
 * X = 2^(floor(log2(amax)) - 8) (8 = the exponent of E4M3's largest normal,
 * 448 = 1.75 * 2^8), clamped to the E8M0 range 2^-127 .. 2^127; each element is
 * E4M3(p / X), rounded to nearest even, with values past 448 saturated.
 * Reading where the specification leaves a choice: a group whose amax is 0
 * gets X = 1 (code 127), as the block-wise scheme uses scale 1 there. */
void oracle_mx_quantise_group(const float* p, uint8_t* q, uint8_t* scale_code)
{
    float amax = 0.0f;
    for (int i = 0; i < ORC_MX_GROUP; ++i) {
        float a = fabsf(p[i]);
        if (a > amax) amax = a;
    }
    int s = 0;
    if (amax > 0.0f) {
        int k = 0;
        (void)frexpf(amax, &k); /* amax = f * 2^k, f in [0.5, 1): floor(log2) = k - 1 */
        s = (k - 1) - 8;
        if (s < -127) s = -127;
        if (s > 127) s = 127;
    }
    *scale_code = (uint8_t)(s + 127);
    float x = ldexpf(1.0f, s);
    for (int i = 0; i < ORC_MX_GROUP; ++i) q[i] = oracle_e4m3_encode(p[i] / x);
}

/* The optimizer step on n_groups consecutive groups of 32 values of a flat
 * row-major shard: the same unscale + clip + AdamW as oracle_step, then the
 * MXFP8 quantiser per group.  Returns 1 (and writes nothing) when found_inf. */
int oracle_mx_step(const orc_hp* hp, double sumsq, int32_t found_inf, const float* grad,
                   float* master, float* m, float* v, uint8_t* codes, uint8_t* scales,
                   int64_t n_groups)
{
    if (found_inf) return 1;
    orc_derived d = derive(hp, sumsq);
    for (int64_t g = 0; g < n_groups; ++g) {
        int64_t base = g * ORC_MX_GROUP;
        for (int64_t i = 0; i < ORC_MX_GROUP; ++i)
            adamw_element(hp, &d, grad[base + i], &master[base + i], &m[base + i], &v[base + i]);
        oracle_mx_quantise_group(master + base, codes + base, &scales[g]);
    }
    return 0;
}
