// Runs the host side of the C ABI (layout and LUT builder, shard ranges, the
// param-wise split, the loss scaler, the clip arithmetic, the MX layout and
// the argument checks) under AddressSanitizer and UndefinedBehaviorSanitizer,
// linked with layout.cpp alone (tests/test_sanitizers.py).  Host-only
// layouts: no device is touched.  Exit status 0 and no report is a pass.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "fp8z1.h"
#include "internal.h"

#define EXPECT(c)                                                     \
    do {                                                              \
        if (!(c)) {                                                   \
            std::fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, #c); \
            return 1;                                                 \
        }                                                             \
    } while (0)

int main()
{
    const std::vector<std::vector<fp8z1_shape>> cases = {
        {{1, 300, 200}},
        {{3, 129, 257}, {1, 1, 1}, {2, 128, 128}, {1, 17, 690}},
        {{32, 7168, 4096}, {32, 2048, 7168}},
        {{1, 2560, 3840}, {1, 300, 200}, {4, 128, 384}, {1, 1000, 131}},
    };
    for (const auto& shapes : cases) {
        const int32_t n = (int32_t)shapes.size();
        for (int32_t dp = 1; dp <= 9; dp += 4) {
            fp8z1_layout* L = nullptr;
            EXPECT(fp8z1_build_layout(shapes.data(), n, dp, FP8Z1_LAYOUT_HOST_ONLY, &L) == FP8Z1_OK);
            int64_t nblk = 0, padded = 0, real = 0;
            EXPECT(fp8z1_layout_info(L, &nblk, &padded, &real) == FP8Z1_OK);
            std::vector<fp8z1_block> lut((size_t)nblk);
            EXPECT(fp8z1_copy_lut(L, lut.data(), nblk) == FP8Z1_OK);
            EXPECT(fp8z1_copy_lut(L, lut.data(), nblk - 1) == FP8Z1_EINVAL);
            int64_t covered = 0;
            for (int32_t r = 0; r < dp; ++r) {
                int64_t b0 = -1, b1 = -1;
                EXPECT(fp8z1_shard_range(L, r, &b0, &b1) == FP8Z1_OK);
                covered += b1 - b0;
            }
            EXPECT(covered == nblk);
            EXPECT(fp8z1_shard_range(L, dp, nullptr, nullptr) == FP8Z1_EINVAL);
            uint32_t bits = 0;
            EXPECT(fp8z1_device_status(L, &bits) == FP8Z1_ENODEV);
            EXPECT(fp8z1_destroy_layout(L) == FP8Z1_OK);

            std::vector<int32_t> owner((size_t)n);
            std::vector<int64_t> bucket((size_t)dp);
            int64_t total = 0;
            EXPECT(fp8z1_paramwise_split(shapes.data(), n, dp, owner.data(), bucket.data(), &total) == FP8Z1_OK);
        }
    }
    // rejected shapes and arguments
    const fp8z1_shape bad[] = {{0, 5, 5}, {1, -1, 5}, {1, 5, (int64_t)1 << 31}, {INT64_MAX, INT64_MAX, 2}};
    for (const auto& s : bad) {
        fp8z1_layout* L = reinterpret_cast<fp8z1_layout*>(1);
        EXPECT(fp8z1_build_layout(&s, 1, 1, FP8Z1_LAYOUT_HOST_ONLY, &L) == FP8Z1_EINVAL && L == nullptr);
    }
    EXPECT(fp8z1_build_layout(nullptr, 1, 1, FP8Z1_LAYOUT_HOST_ONLY, nullptr) == FP8Z1_EINVAL);
    EXPECT(fp8z1_destroy_layout(nullptr) == FP8Z1_OK);

    // loss scaler and clip arithmetic
    fp8z1_loss_scaler sc = {65536.0f, 0, 0, 2};
    for (int i = 0; i < 10; ++i) EXPECT(fp8z1_scaler_update(&sc, i % 4 == 3) == FP8Z1_OK);
    EXPECT(fp8z1_scaler_update(nullptr, 0) == FP8Z1_EINVAL);
    double gn = 0, cc = 0;
    EXPECT(fp8z1_clip_coef(4.0e6, 1.0f, 1024.0f, &gn, &cc) == FP8Z1_OK);
    EXPECT(fp8z1_clip_coef(0.0, 1.0f, 1024.0f, &gn, &cc) == FP8Z1_OK);

    // the MX layout (every C a multiple of 32)
    const fp8z1_shape mx[] = {{32, 7168, 4096}, {1, 300, 64}, {2, 3, 32}};
    fp8z1_mx_layout* M = nullptr;
    EXPECT(fp8z1_mx_build_layout(mx, 3, 8, FP8Z1_LAYOUT_HOST_ONLY, &M) == FP8Z1_OK);
    int64_t ng = 0, ne = 0, cov = 0;
    EXPECT(fp8z1_mx_layout_info(M, &ng, &ne) == FP8Z1_OK);
    for (int32_t r = 0; r < 8; ++r) {
        int64_t g0, g1;
        EXPECT(fp8z1_mx_shard_range(M, r, &g0, &g1) == FP8Z1_OK);
        cov += g1 - g0;
    }
    EXPECT(cov == ng);
    EXPECT(fp8z1_mx_destroy_layout(M) == FP8Z1_OK);
    const fp8z1_shape mx_bad = {1, 4, 33};
    EXPECT(fp8z1_mx_build_layout(&mx_bad, 1, 1, FP8Z1_LAYOUT_HOST_ONLY, &M) == FP8Z1_EINVAL);

    // the pieces of a grad norm without store: for every sub-range [b0, b1),
    // every real element of its blocks exactly once, nothing else
    const std::vector<std::vector<fp8z1_shape>> small = {
        {{1, 300, 200}},
        {{3, 129, 257}, {1, 1, 1}, {2, 128, 128}, {1, 17, 690}},
        {{2, 300, 260}, {1, 200, 131}, {2, 256, 256}},
    };
    std::vector<fp8z1::NormPiece> pieces;
    for (const auto& shapes : small) {
        const int32_t n = (int32_t)shapes.size();
        fp8z1_layout* L = nullptr;
        EXPECT(fp8z1_build_layout(shapes.data(), n, 1, FP8Z1_LAYOUT_HOST_ONLY, &L) == FP8Z1_OK);
        const int64_t nblk = L->n_blocks;
        std::vector<std::vector<uint8_t>> got(shapes.size()), want(shapes.size());
        for (int64_t b0 = 0; b0 <= nblk; ++b0)
            for (int64_t b1 = b0; b1 <= nblk; ++b1) {
                for (int32_t i = 0; i < n; ++i) {
                    const size_t ne = (size_t)(shapes[i].E * shapes[i].R * shapes[i].C);
                    got[i].assign(ne, 0);
                    want[i].assign(ne, 0);
                }
                auto mark_block = [&](std::vector<std::vector<uint8_t>>& cov, int64_t k) {
                    const fp8z1_block& blk = L->lut[(size_t)k];
                    for (int r = 0; r < blk.rows_real; ++r)
                        for (int c = 0; c < blk.cols_real; ++c)
                            ++cov[blk.param][(size_t)(blk.src_offset + (int64_t)r * blk.ld + c)];
                };
                for (int64_t k = b0; k < b1; ++k) mark_block(want, k);
                fp8z1::norm_pieces(L, b0, b1, pieces);
                for (const auto& pc : pieces) {
                    if (pc.kind == fp8z1::NormPiece::kBlocks) {
                        EXPECT(pc.a < pc.b);
                        for (int64_t k = pc.a; k < pc.b; ++k) mark_block(got, k);
                    } else if (pc.kind == fp8z1::NormPiece::kWholeParams) {
                        EXPECT(pc.a < pc.b);
                        for (int64_t q = pc.a; q < pc.b; ++q)
                            for (auto& x : got[(size_t)q]) ++x;
                    } else {
                        EXPECT(pc.a < pc.b && pc.b <= (int64_t)got[(size_t)pc.param].size());
                        for (int64_t e = pc.a; e < pc.b; ++e) ++got[(size_t)pc.param][(size_t)e];
                    }
                }
                EXPECT(got == want);
                for (const auto& v : got)
                    for (uint8_t x : v) EXPECT(x <= 1);
                EXPECT(pieces.size() <= 4 || b1 - b0 > 2);
            }
        EXPECT(fp8z1_destroy_layout(L) == FP8Z1_OK);
    }

    uint64_t launches = 1;
    EXPECT(fp8z1_kernel_launches(&launches) == FP8Z1_OK && launches == 0);
    // the release build's checked-build entry points: flags 0, no misses, no table hook
    EXPECT(fp8z1_build_flags() == 0);
    uint64_t misses = 7;
    EXPECT(fp8z1_checked_misses(&misses) == FP8Z1_OK && misses == 0);
    EXPECT(fp8z1_checked_misses(nullptr) == FP8Z1_EINVAL);
    {
        const fp8z1_shape one = {1, 128, 128};
        fp8z1_layout* L = nullptr;
        EXPECT(fp8z1_build_layout(&one, 1, 1, FP8Z1_LAYOUT_HOST_ONLY, &L) == FP8Z1_OK);
        fp8z1_block e = {};
        EXPECT(fp8z1_checked_set_lut_entry(L, 0, &e) == FP8Z1_EINVAL);
        EXPECT(fp8z1_destroy_layout(L) == FP8Z1_OK);
    }
    for (int st = 1; st >= -9; --st) EXPECT(fp8z1_strerror(st) != nullptr);
    std::printf("layout driver ok\n");
    return 0;
}
