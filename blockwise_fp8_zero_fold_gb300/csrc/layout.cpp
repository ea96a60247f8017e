// Host side of libfp8z1.so: the block lookup table, shard ranges, the loss
// scaler and status text.
//
// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §块粒度切分: each quantised dim
// is padded up to a multiple of 128, a lookup table records every 128x128
// block's param and real extent, and ZeRO shards are cut on block edges;
// §参数布局变换: block order of fold is (expert, row block, col block).
#include <limits.h>
#include <math.h>

#include <algorithm>
#include <new>

#include "internal.h"

namespace {

constexpr int64_t kTile = FP8Z1_TILE;

int64_t tiles(int64_t n) { return (n + kTile - 1) / kTile; }

// Free whatever device memory a layout holds (safe on partial layouts).
void release_device(fp8z1_layout* L)
{
    cudaFree(L->d_lut);
    cudaFree(L->d_units);
    cudaFree(L->d_param_elems);
    cudaFree(L->d_partials);
    cudaFree(L->d_counter);
    cudaFree(L->d_status);
    L->d_lut = nullptr;
    L->d_units = nullptr;
    L->d_param_elems = nullptr;
    L->d_partials = nullptr;
    L->d_counter = nullptr;
    L->d_status = nullptr;
}

int upload(fp8z1_layout* L)
{
    if (cudaGetDevice(&L->device) != cudaSuccess) return FP8Z1_ECUDA;
    if (cudaDeviceGetAttribute(&L->sm_count, cudaDevAttrMultiProcessorCount, L->device) != cudaSuccess)
        return FP8Z1_ECUDA;
    // grad-norm workspace: up to 4 CTAs per SM, capped at 4096 partial sums
    L->max_partials = L->sm_count * 4 < 4096 ? L->sm_count * 4 : 4096;
    const size_t lut_bytes = sizeof(fp8z1_block) * (size_t)L->n_blocks;
    const size_t unit_bytes = sizeof(fp8z1_unit) * L->units.size();
    std::vector<int64_t> elems;
    try {
        elems.resize(L->shapes.size());
    } catch (...) {
        return FP8Z1_ENOMEM;
    }
    for (size_t i = 0; i < L->shapes.size(); ++i) elems[i] = L->shapes[i].E * L->shapes[i].R * L->shapes[i].C;
    const size_t elems_bytes = sizeof(int64_t) * elems.size();
    if (cudaMalloc(&L->d_lut, lut_bytes ? lut_bytes : sizeof(fp8z1_block)) != cudaSuccess ||
        cudaMalloc(&L->d_units, unit_bytes ? unit_bytes : sizeof(fp8z1_unit)) != cudaSuccess ||
        cudaMalloc(&L->d_param_elems, elems_bytes ? elems_bytes : sizeof(int64_t)) != cudaSuccess ||
        cudaMalloc(&L->d_partials, sizeof(double) * (size_t)L->max_partials) != cudaSuccess ||
        cudaMalloc(&L->d_counter, sizeof(unsigned)) != cudaSuccess ||
        cudaMalloc(&L->d_status, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ENOMEM;
    }
    if (lut_bytes && cudaMemcpy(L->d_lut, L->lut.data(), lut_bytes, cudaMemcpyHostToDevice) != cudaSuccess)
        return FP8Z1_ECUDA;
    if (unit_bytes && cudaMemcpy(L->d_units, L->units.data(), unit_bytes, cudaMemcpyHostToDevice) != cudaSuccess)
        return FP8Z1_ECUDA;
    if (elems_bytes && cudaMemcpy(L->d_param_elems, elems.data(), elems_bytes, cudaMemcpyHostToDevice) != cudaSuccess)
        return FP8Z1_ECUDA;
    if (cudaMemset(L->d_counter, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(L->d_status, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return FP8Z1_ECUDA;
    L->on_device = true;
    return FP8Z1_OK;
}

}  // namespace

extern "C" int fp8z1_build_layout(const fp8z1_shape* shapes, int32_t n_params, int32_t dp_size,
                                  uint32_t flags, fp8z1_layout** out)
{
    if (!out) return FP8Z1_EINVAL;
    *out = nullptr;
    if (!shapes || n_params < 1 || dp_size < 1 || (flags & ~FP8Z1_LAYOUT_HOST_ONLY)) return FP8Z1_EINVAL;
    // validate shapes and count blocks without overflowing int64
    int64_t nblk = 0, nreal = 0;
    const int64_t kMax = INT64_MAX / FP8Z1_BLOCK_ELEMS;
    for (int32_t i = 0; i < n_params; ++i) {
        const fp8z1_shape s = shapes[i];
        if (s.E < 1 || s.R < 1 || s.C < 1 || s.C > INT_MAX || s.E > INT_MAX || tiles(s.R) > INT_MAX)
            return FP8Z1_EINVAL;
        const int64_t rb = tiles(s.R), cb = tiles(s.C);
        if (rb > kMax / cb || s.E > kMax / (rb * cb)) return FP8Z1_EINVAL;
        const int64_t nb = s.E * rb * cb;
        if (nb > kMax - nblk) return FP8Z1_EINVAL;
        nblk += nb;
        nreal += s.E * s.R * s.C;  // <= padded count, which fits
    }
    fp8z1_layout* L = new (std::nothrow) fp8z1_layout();
    if (!L) return FP8Z1_ENOMEM;
    try {
        L->shapes.assign(shapes, shapes + n_params);
        L->lut.resize((size_t)nblk);
    } catch (...) {
        delete L;
        return FP8Z1_ENOMEM;
    }
    L->n_params = n_params;
    L->dp_size = dp_size;
    L->n_blocks = nblk;
    L->n_real = nreal;
    int64_t k = 0;
    for (int32_t i = 0; i < n_params; ++i) {
        const fp8z1_shape s = shapes[i];
        const int64_t rbs = tiles(s.R), cbs = tiles(s.C);
        for (int64_t e = 0; e < s.E; ++e)
            for (int64_t rb = 0; rb < rbs; ++rb)
                for (int64_t cb = 0; cb < cbs; ++cb) {
                    fp8z1_block& b = L->lut[(size_t)k++];
                    b.src_offset = (e * s.R + kTile * rb) * s.C + kTile * cb;
                    b.param = i;
                    b.expert = (int32_t)e;
                    b.row_block = (int32_t)rb;
                    b.col_block = (int32_t)cb;
                    b.ld = (int32_t)s.C;
                    const int64_t rr = s.R - kTile * rb, cr = s.C - kTile * cb;
                    b.rows_real = (int16_t)(rr < kTile ? rr : kTile);
                    b.cols_real = (int16_t)(cr < kTile ? cr : kTile);
                }
    }
    // runs of params made of full tiles only (the step skips no padding there)
    try {
        // each param's first block, and its row-major elements cut into units
        L->param_block0.resize((size_t)n_params + 1);
        L->param_unit0.resize((size_t)n_params + 1);
        int64_t nunits = 0;
        for (int32_t i = 0; i < n_params; ++i)
            nunits += (shapes[i].E * shapes[i].R * shapes[i].C + FP8Z1_BLOCK_ELEMS - 1) / FP8Z1_BLOCK_ELEMS;
        L->units.reserve((size_t)nunits);
        int64_t b = 0;
        for (int32_t i = 0; i < n_params; ++i) {
            L->param_block0[(size_t)i] = b;
            L->param_unit0[(size_t)i] = (int64_t)L->units.size();
            b += shapes[i].E * tiles(shapes[i].R) * tiles(shapes[i].C);
            const int64_t n = shapes[i].E * shapes[i].R * shapes[i].C;
            for (int64_t o = 0; o < n; o += FP8Z1_BLOCK_ELEMS)
                L->units.push_back({o, i, (int32_t)(n - o < FP8Z1_BLOCK_ELEMS ? n - o : FP8Z1_BLOCK_ELEMS)});
        }
        L->param_block0[(size_t)n_params] = b;
        L->param_unit0[(size_t)n_params] = (int64_t)L->units.size();
        int64_t first = 0, run0 = -1;
        for (int32_t i = 0; i <= n_params; ++i) {
            const bool full = i < n_params && shapes[i].R % kTile == 0 && shapes[i].C % kTile == 0;
            if (full && run0 < 0) run0 = first;
            if (!full && run0 >= 0) {
                if (first - run0 >= fp8z1_layout::kFullRunMin) {
                    L->full_runs.push_back(run0);
                    L->full_runs.push_back(first);
                }
                run0 = -1;
            }
            if (i < n_params) first += shapes[i].E * tiles(shapes[i].R) * tiles(shapes[i].C);
        }
    } catch (...) {
        delete L;
        return FP8Z1_ENOMEM;
    }
    if (!(flags & FP8Z1_LAYOUT_HOST_ONLY)) {
        const int st = upload(L);
        if (st != FP8Z1_OK) {
            release_device(L);
            delete L;
            return st;
        }
    }
    *out = L;
    return FP8Z1_OK;
}

void fp8z1::norm_pieces(const fp8z1_layout* L, int64_t b0, int64_t b1, std::vector<NormPiece>& out)
{
    out.clear();
    auto add_blocks = [&](int64_t k0, int64_t k1) {
        if (k0 == k1) return;
        if (!out.empty() && out.back().kind == NormPiece::kBlocks && out.back().b == k0)
            out.back().b = k1;  // adjacent block ranges: one launch
        else
            out.push_back({NormPiece::kBlocks, k0, k1, 0});
    };
    const std::vector<int64_t>& pb = L->param_block0;
    int64_t p = std::upper_bound(pb.begin(), pb.end(), b0) - pb.begin() - 1;  // the param holding block b0
    for (; b0 < b1 && p < L->n_params && pb[(size_t)p] < b1; ++p) {
        const int64_t k0 = std::max(pb[(size_t)p], b0), k1 = std::min(pb[(size_t)p + 1], b1);
        if (k0 == pb[(size_t)p] && k1 == pb[(size_t)p + 1]) {  // held whole
            if (!out.empty() && out.back().kind == NormPiece::kWholeParams && out.back().b == p)
                out.back().b = p + 1;
            else
                out.push_back({NormPiece::kWholeParams, p, p + 1, 0});
            continue;
        }
        const fp8z1_shape sh = L->shapes[(size_t)p];
        const int64_t rbs = tiles(sh.R), cbs = tiles(sh.C);
        const int64_t l0 = k0 - pb[(size_t)p], l1 = k1 - pb[(size_t)p];
        const int64_t s0 = (l0 + cbs - 1) / cbs, s1 = l1 / cbs;  // the whole strips [s0, s1)
        if (s0 >= s1) {
            add_blocks(k0, k1);
            continue;
        }
        // strip s = e * rbs + rb starts at row e * R + 128 rb; strip E * rbs ends the param
        auto strip_elem = [&](int64_t st) {
            return st == sh.E * rbs ? sh.E * sh.R * sh.C : ((st / rbs) * sh.R + (st % rbs) * kTile) * sh.C;
        };
        add_blocks(k0, pb[(size_t)p] + s0 * cbs);
        out.push_back({NormPiece::kSpan, strip_elem(s0), strip_elem(s1), (int32_t)p});
        add_blocks(pb[(size_t)p] + s1 * cbs, k1);
    }
}

std::atomic<uint64_t>& fp8z1::launch_counter()
{
    static std::atomic<uint64_t> n{0};
    return n;
}

extern "C" int fp8z1_kernel_launches(uint64_t* out)
{
    if (!out) return FP8Z1_EINVAL;
    *out = fp8z1::launch_counter().load(std::memory_order_relaxed);
    return FP8Z1_OK;
}

extern "C" int fp8z1_build_flags(void)
{
    return FP8Z1_CHECKED ? FP8Z1_BUILD_CHECKED : 0;
}

extern "C" int fp8z1_checked_misses(uint64_t* count)
{
    if (!count) return FP8Z1_EINVAL;
    *count = 0;
#if FP8Z1_CHECKED
    const uint64_t parts[] = {fp8z1::checked_misses_fold(), fp8z1::checked_misses_norm(),
                              fp8z1::checked_misses_step_full(), fp8z1::checked_misses_step_pad()};
    for (uint64_t v : parts) {
        if (v == ~0ull) return FP8Z1_ECUDA;
        *count += v;
    }
#endif
    return FP8Z1_OK;
}

extern "C" int fp8z1_checked_set_lut_entry(fp8z1_layout* L, int64_t block, const fp8z1_block* entry)
{
#if FP8Z1_CHECKED
    if (!L || !entry || block < 0 || block >= L->n_blocks) return FP8Z1_EINVAL;
    if (!L->on_device) return FP8Z1_ENODEV;
    if (cudaMemcpy(L->d_lut + block, entry, sizeof(fp8z1_block), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return FP8Z1_ECUDA;
    }
    return FP8Z1_OK;
#else
    (void)L;
    (void)block;
    (void)entry;
    return FP8Z1_EINVAL;
#endif
}

extern "C" int fp8z1_destroy_layout(fp8z1_layout* L)
{
    if (!L) return FP8Z1_OK;
    if (L->on_device) release_device(L);
    delete L;
    return FP8Z1_OK;
}

extern "C" int fp8z1_layout_info(const fp8z1_layout* L, int64_t* n_blocks, int64_t* n_elems_padded,
                                 int64_t* n_elems_real)
{
    if (!L) return FP8Z1_EINVAL;
    if (n_blocks) *n_blocks = L->n_blocks;
    if (n_elems_padded) *n_elems_padded = L->n_blocks * FP8Z1_BLOCK_ELEMS;
    if (n_elems_real) *n_elems_real = L->n_real;
    return FP8Z1_OK;
}

extern "C" int fp8z1_shard_range(const fp8z1_layout* L, int32_t rank, int64_t* b0, int64_t* b1)
{
    if (!L || !b0 || !b1 || rank < 0 || rank >= L->dp_size) return FP8Z1_EINVAL;
    const int64_t per = (L->n_blocks + L->dp_size - 1) / L->dp_size;
    int64_t lo = per * rank, hi = per * (rank + 1);
    *b0 = lo < L->n_blocks ? lo : L->n_blocks;
    *b1 = hi < L->n_blocks ? hi : L->n_blocks;
    return FP8Z1_OK;
}

extern "C" int fp8z1_copy_lut(const fp8z1_layout* L, fp8z1_block* host_dst, int64_t capacity)
{
    if (!L || (!host_dst && L->n_blocks) || capacity < L->n_blocks) return FP8Z1_EINVAL;
    for (int64_t k = 0; k < L->n_blocks; ++k) host_dst[k] = L->lut[(size_t)k];
    return FP8Z1_OK;
}

// §总结 ends by unfolding the 1-D blockwise scales into each param's 2-D / 3-D
// scales.  Blocks run param by param and, inside a param, in (e, rb, cb)
// row-major order (§参数布局变换), so a param's scales are one contiguous
// [E, ceil(R/128), ceil(C/128)] stretch of the scale buffer; this reports
// where it starts and which experts of it a block range holds whole.
extern "C" int fp8z1_param_blocks(const fp8z1_layout* L, int32_t param, int64_t b0, int64_t b1,
                                  fp8z1_param_grid* out)
{
    if (!L || !out || param < 0 || param >= L->n_params) return FP8Z1_EINVAL;
    if (b0 < 0 || b1 < b0 || b1 > L->n_blocks) return FP8Z1_EINVAL;
    const fp8z1_shape& sh = L->shapes[(size_t)param];
    fp8z1_param_grid g;
    g.first_block = L->param_block0[(size_t)param];
    g.experts = sh.E;
    g.row_blocks = tiles(sh.R);
    g.col_blocks = tiles(sh.C);
    const int64_t per = g.row_blocks * g.col_blocks;  // blocks of one expert
    // experts e with [first + e*per, first + (e+1)*per) inside [b0, b1)
    int64_t lo = b0 - g.first_block, hi = b1 - g.first_block;
    int64_t e0 = lo <= 0 ? 0 : (lo + per - 1) / per;
    int64_t e1 = hi <= 0 ? 0 : hi / per;
    if (e0 > g.experts) e0 = g.experts;
    if (e1 > g.experts) e1 = g.experts;
    if (e1 < e0) e1 = e0;
    g.e_begin = e0;
    g.e_end = e1;
    *out = g;
    return FP8Z1_OK;
}

extern "C" int fp8z1_device_status(const fp8z1_layout* L, uint32_t* bits)
{
    if (!L || !bits) return FP8Z1_EINVAL;
    if (!L->on_device) return FP8Z1_ENODEV;
    unsigned v = 0;
    if (cudaMemcpy(&v, L->d_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(L->d_status, 0, sizeof v) != cudaSuccess)
        return FP8Z1_ECUDA;
    *bits = v;
    return FP8Z1_OK;
}

// "DeepSpeed ZeRO 优化" §六 Loss Scaling: an overflow halves S and skips the
// step; N clean steps in a row double S.
extern "C" int fp8z1_scaler_update(fp8z1_loss_scaler* s, int32_t found_inf)
{
    if (!s || !(s->scale > 0.0f) || s->growth_interval < 1) return FP8Z1_EINVAL;
    if (found_inf) {
        s->scale *= 0.5f;
        s->good_steps = 0;
        return FP8Z1_OK;
    }
    s->step += 1;
    if (++s->good_steps >= s->growth_interval) {
        s->scale *= 2.0f;
        s->good_steps = 0;
    }
    return FP8Z1_OK;
}

// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §参数粒度切分: the page's other
// split.  Params sorted by size, largest first (equal sizes keep their order),
// each given to the DP bucket with the fewest elements so far (the lowest
// index on a tie); every bucket is then padded to the largest.
extern "C" int fp8z1_paramwise_split(const fp8z1_shape* shapes, int32_t n_params, int32_t dp_size,
                                     int32_t* owner, int64_t* bucket_elems, int64_t* padded_total)
{
    if (!shapes || n_params < 1 || dp_size < 1 || !owner || !bucket_elems) return FP8Z1_EINVAL;
    std::vector<int64_t> size((size_t)n_params);
    for (int32_t i = 0; i < n_params; ++i) {
        const fp8z1_shape s = shapes[i];
        if (s.E < 1 || s.R < 1 || s.C < 1 || s.R > INT64_MAX / s.C || s.E > INT64_MAX / (s.R * s.C))
            return FP8Z1_EINVAL;
        size[(size_t)i] = s.E * s.R * s.C;
    }
    std::vector<int32_t> order((size_t)n_params);
    for (int32_t i = 0; i < n_params; ++i) order[(size_t)i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return size[(size_t)a] > size[(size_t)b]; });
    for (int32_t b = 0; b < dp_size; ++b) bucket_elems[b] = 0;
    for (int32_t i : order) {
        int32_t best = 0;
        for (int32_t b = 1; b < dp_size; ++b)
            if (bucket_elems[b] < bucket_elems[best]) best = b;
        owner[i] = best;
        bucket_elems[best] += size[(size_t)i];
    }
    if (padded_total) {
        int64_t mx = 0;
        for (int32_t b = 0; b < dp_size; ++b) mx = bucket_elems[b] > mx ? bucket_elems[b] : mx;
        *padded_total = mx * dp_size;
    }
    return FP8Z1_OK;
}

// "DeepSpeed ZeRO 优化" §七: the clip arithmetic the step kernels perform on
// the device, on the host, for logging.
extern "C" int fp8z1_clip_coef(double sumsq, float max_norm, float loss_scale, double* global_norm,
                               double* clip_coef)
{
    if (!global_norm || !clip_coef || !(loss_scale > 0.0f) || !(max_norm > 0.0f) || !(sumsq >= 0.0))
        return FP8Z1_EINVAL;
    *global_norm = sqrt(sumsq) / (double)loss_scale;
    *clip_coef = (double)max_norm / (*global_norm + 1e-6);
    return FP8Z1_OK;
}

// ---- MXFP8 layout --------------------------------------------------------

extern "C" int fp8z1_mx_build_layout(const fp8z1_shape* shapes, int32_t n_params, int32_t dp_size,
                                     uint32_t flags, fp8z1_mx_layout** out)
{
    if (!out) return FP8Z1_EINVAL;
    *out = nullptr;
    if (!shapes || n_params < 1 || dp_size < 1 || (flags & ~FP8Z1_LAYOUT_HOST_ONLY)) return FP8Z1_EINVAL;
    int64_t groups = 0;
    const int64_t kMax = INT64_MAX / FP8Z1_MX_GROUP;
    for (int32_t i = 0; i < n_params; ++i) {
        const fp8z1_shape s = shapes[i];
        if (s.E < 1 || s.R < 1 || s.C < 1 || s.C % FP8Z1_MX_GROUP != 0) return FP8Z1_EINVAL;
        const int64_t per_row = s.C / FP8Z1_MX_GROUP;
        if (s.R > kMax / per_row || s.E > kMax / (s.R * per_row)) return FP8Z1_EINVAL;
        const int64_t g = s.E * s.R * per_row;
        if (g > kMax - groups) return FP8Z1_EINVAL;
        groups += g;
    }
    fp8z1_mx_layout* L = new (std::nothrow) fp8z1_mx_layout();
    if (!L) return FP8Z1_ENOMEM;
    try {
        L->shapes.assign(shapes, shapes + n_params);
    } catch (...) {
        delete L;
        return FP8Z1_ENOMEM;
    }
    L->n_params = n_params;
    L->dp_size = dp_size;
    L->n_groups = groups;
    if (!(flags & FP8Z1_LAYOUT_HOST_ONLY)) {
        int dev = 0;
        int st = FP8Z1_OK;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&L->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            st = FP8Z1_ECUDA;
        if (st == FP8Z1_OK) {
            L->max_partials = L->sm_count * 4 < 4096 ? L->sm_count * 4 : 4096;
            if (cudaMalloc(&L->d_partials, sizeof(double) * (size_t)L->max_partials) != cudaSuccess ||
                cudaMalloc(&L->d_counter, sizeof(unsigned)) != cudaSuccess)
                st = FP8Z1_ENOMEM;
            else if (cudaMemset(L->d_counter, 0, sizeof(unsigned)) != cudaSuccess ||
                     cudaDeviceSynchronize() != cudaSuccess)
                st = FP8Z1_ECUDA;
        }
        if (st != FP8Z1_OK) {
            cudaGetLastError();
            cudaFree(L->d_partials);
            cudaFree(L->d_counter);
            delete L;
            return st;
        }
        L->on_device = true;
    }
    *out = L;
    return FP8Z1_OK;
}

extern "C" int fp8z1_mx_destroy_layout(fp8z1_mx_layout* L)
{
    if (!L) return FP8Z1_OK;
    if (L->on_device) {
        cudaFree(L->d_partials);
        cudaFree(L->d_counter);
    }
    delete L;
    return FP8Z1_OK;
}

extern "C" int fp8z1_mx_layout_info(const fp8z1_mx_layout* L, int64_t* n_groups, int64_t* n_elems)
{
    if (!L) return FP8Z1_EINVAL;
    if (n_groups) *n_groups = L->n_groups;
    if (n_elems) *n_elems = L->n_groups * FP8Z1_MX_GROUP;
    return FP8Z1_OK;
}

extern "C" int fp8z1_mx_shard_range(const fp8z1_mx_layout* L, int32_t rank, int64_t* g0, int64_t* g1)
{
    if (!L || !g0 || !g1 || rank < 0 || rank >= L->dp_size) return FP8Z1_EINVAL;
    const int64_t per = (L->n_groups + L->dp_size - 1) / L->dp_size;
    const int64_t lo = per * rank, hi = per * (rank + 1);
    *g0 = lo < L->n_groups ? lo : L->n_groups;
    *g1 = hi < L->n_groups ? hi : L->n_groups;
    return FP8Z1_OK;
}

extern "C" const char* fp8z1_strerror(int status)
{
    switch (status) {
    case FP8Z1_OK: return "ok";
    case FP8Z1_EINVAL: return "invalid argument";
    case FP8Z1_EALIGN: return "misaligned pointer";
    case FP8Z1_ENOMEM: return "out of memory";
    case FP8Z1_ECUDA: return "CUDA runtime error";
    case FP8Z1_ENODEV: return "layout has no device tables (built host-only)";
    default: return "unknown status";
    }
}
