// fold / unfold: the mutually inverse layout transforms between row-major
// [E, R, C] params and the 128x128-block-contiguous 1-D buffer.
//
// "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §参数布局变换: fold is
// view(E, R/128, 128, C/128, 128).permute(0, 1, 3, 2, 4) made contiguous, so
// each 128-element row segment of a block stays contiguous on both sides;
// §块粒度切分: R and C are zero-padded up to multiples of 128.
//
// A CTA copies a run of BPC consecutive 128x128 blocks, one after the other;
// each block's source rows are found through the lookup table (param, element
// offset, row stride, real extent), the next block's entry and param pointer
// loaded while the current block is copied.  When the
// param's row stride and base are 16-byte aligned, every 16-byte chunk of a
// block row is either all real or all padding (real columns * elem_size is
// then a multiple of 16), so the copy moves 16-byte vectors: coalesced on the
// block side (contiguous) and on the row-major side (a row segment is 128 *
// elem_size contiguous bytes).  Otherwise each thread moves single elements,
// still coalesced along rows.
#include "checked.cuh"

namespace {

constexpr int kThreads = 256;

template <int ESZ> struct ElemT;
template <> struct ElemT<1> { using T = uint8_t; };
template <> struct ElemT<2> { using T = uint16_t; };
template <> struct ElemT<4> { using T = uint32_t; };

__device__ __forceinline__ uint4 ld_stream16(const uint8_t* p)
{
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st_stream16(uint8_t* p, uint4 v)
{
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// Copy one block between its row-major tile and its place buf in the shard.
// elems: the param's extent, against which a checked build tests each access.
template <int ESZ, bool FOLD>
__device__ __forceinline__ void copy_block(const fp8z1_block& blk, uint8_t* base, uint8_t* buf, int64_t elems)
{
    using T = typename ElemT<ESZ>::T;
    uint8_t* const tile = base + blk.src_offset * ESZ;
    const int64_t ld = (int64_t)blk.ld * ESZ;  // row stride in bytes
    const int rows = blk.rows_real, cols = blk.cols_real;

    if (((ld | reinterpret_cast<intptr_t>(tile)) & 15) == 0) {
        constexpr int kVPR = FP8Z1_TILE * ESZ / 16;        // 16-byte vectors per block row
        constexpr int kIters = FP8Z1_TILE * kVPR / kThreads;  // 16, 8, 4
        constexpr int kU = kIters < 8 ? kIters : 8;          // vectors in flight per thread
        const int cv = cols * ESZ / 16;                      // real vectors per row
#pragma unroll 1
        for (int j0 = 0; j0 < kIters; j0 += kU) {
            uint4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = threadIdx.x + (j0 + u) * kThreads;
                const int r = i / kVPR, c = i % kVPR;
                const bool real = r < rows && c < cv;
                if (FOLD)
                    v[u] = real && fp8z1::in_extent(blk.src_offset + (int64_t)r * blk.ld + c * (16 / ESZ), 16 / ESZ,
                                                    elems)
                               ? ld_stream16(tile + r * ld + c * 16)
                               : make_uint4(0, 0, 0, 0);
                else if (real)
                    v[u] = ld_stream16(buf + (int64_t)i * 16);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = threadIdx.x + (j0 + u) * kThreads;
                const int r = i / kVPR, c = i % kVPR;
                if (FOLD)
                    st_stream16(buf + (int64_t)i * 16, v[u]);
                else if (r < rows && c < cv &&
                         fp8z1::in_extent(blk.src_offset + (int64_t)r * blk.ld + c * (16 / ESZ), 16 / ESZ, elems))
                    st_stream16(tile + r * ld + c * 16, v[u]);
            }
        }
    } else {
        constexpr int kIters = FP8Z1_BLOCK_ELEMS / kThreads;  // 64
        constexpr int kU = 16;
#pragma unroll 1
        for (int j0 = 0; j0 < kIters; j0 += kU) {
            T v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = threadIdx.x + (j0 + u) * kThreads;
                const int r = i / FP8Z1_TILE, c = i % FP8Z1_TILE;
                const bool real = r < rows && c < cols;
                if (FOLD)
                    v[u] = real && fp8z1::in_extent(blk.src_offset + (int64_t)r * blk.ld + c, 1, elems)
                               ? reinterpret_cast<const T*>(tile + r * ld)[c]
                               : T(0);
                else if (real)
                    v[u] = reinterpret_cast<const T*>(buf)[i];
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = threadIdx.x + (j0 + u) * kThreads;
                const int r = i / FP8Z1_TILE, c = i % FP8Z1_TILE;
                if (FOLD)
                    reinterpret_cast<T*>(buf)[i] = v[u];
                else if (r < rows && c < cols && fp8z1::in_extent(blk.src_offset + (int64_t)r * blk.ld + c, 1, elems))
                    reinterpret_cast<T*>(tile + r * ld)[c] = v[u];
            }
        }
    }
}

// Blocks b0 + [BPC x, BPC x + BPC) of the range (x = blockIdx.x), clipped to
// its n blocks.  A block whose param pointer is null or misaligned is left
// untouched and reported in *status.  3 CTAs per SM (2 for the 2- and 4-byte
// unfolds, whose two copy paths together need about 128 registers unspilled).
template <int ESZ, bool FOLD, int BPC>
__global__ void __launch_bounds__(kThreads, (FOLD || ESZ == 1) ? 3 : 2) fold_kernel(const fp8z1_block* __restrict__ lut,
                                                        void* const* __restrict__ params,
                                                        uint8_t* __restrict__ shard, int64_t b0, int64_t n,
                                                        unsigned* __restrict__ status,
                                                        const int64_t* __restrict__ param_elems)
{
    const int64_t k0 = (int64_t)blockIdx.x * BPC;
    const int64_t k1 = k0 + BPC < n ? k0 + BPC : n;
    fp8z1_block blk = lut[b0 + k0];
    uint8_t* base = static_cast<uint8_t*>(params[blk.param]);
    for (int64_t k = k0; k < k1; ++k) {
        fp8z1_block next = blk;
        uint8_t* next_base = nullptr;
        if (k + 1 < k1) {
            next = lut[b0 + k + 1];
            next_base = static_cast<uint8_t*>(params[next.param]);
        }
        if (base == nullptr || (reinterpret_cast<uintptr_t>(base) % ESZ) != 0) {
            if (threadIdx.x == 0) atomicOr(status, FP8Z1_DEV_BADPTR);
        } else {
            const int64_t elems = FP8Z1_CHECKED ? param_elems[blk.param] : 0;
            copy_block<ESZ, FOLD>(blk, base, shard + k * (FP8Z1_BLOCK_ELEMS * ESZ), elems);
        }
        blk = next;
        base = next_base;
    }
}

// Blocks per CTA: one for the folds; four for the 1- and 2-byte unfolds, which
// gained 1-1.5% from it (MoE buffer, back to back: FP8 codes 0.418 -> 0.412
// ms, bf16 0.810 -> 0.800 ms); the folds lost 1-2% from more than one.
constexpr int kBpcUnfoldNarrow = 4;

template <int ESZ, bool FOLD, int BPC>
void launch_esz(const fp8z1_layout* L, void* const* params, uint8_t* shard, int64_t b0, int64_t n,
                cudaStream_t stream)
{
    const dim3 grid((unsigned)((n + BPC - 1) / BPC)), block(kThreads);
    fold_kernel<ESZ, FOLD, BPC><<<grid, block, 0, stream>>>(L->d_lut, params, shard, b0, n, L->d_status,
                                                          L->d_param_elems);
}

template <bool FOLD>
int launch(const fp8z1_layout* L, void* const* params, uint8_t* shard, int32_t esz, int64_t b0,
           int64_t b1, cudaStream_t stream)
{
    const int64_t n = b1 - b0;
    fp8z1::count_launch();
    constexpr int kNarrow = FOLD ? 1 : kBpcUnfoldNarrow;
    switch (esz) {
    case 1: launch_esz<1, FOLD, kNarrow>(L, params, shard, b0, n, stream); break;
    case 2: launch_esz<2, FOLD, kNarrow>(L, params, shard, b0, n, stream); break;
    default: launch_esz<4, FOLD, 1>(L, params, shard, b0, n, stream); break;
    }
    return fp8z1::launch_status();
}

int check(const fp8z1_layout* L, const void* params, const void* shard, int32_t esz, int64_t b0,
          int64_t b1)
{
    if (!params || !shard || (esz != 1 && esz != 2 && esz != 4)) return FP8Z1_EINVAL;
    const int st = fp8z1::check_range(L, b0, b1);
    if (st != FP8Z1_OK) return st;
    if (b1 - b0 > 0x7fffffffLL) return FP8Z1_EINVAL;  // one CTA per block
    if (!fp8z1::aligned(shard, 16) || !fp8z1::aligned(params, sizeof(void*))) return FP8Z1_EALIGN;
    return FP8Z1_OK;
}

}  // namespace

extern "C" int fp8z1_fold(const fp8z1_layout* L, const void* const* d_src_params, void* dst_shard,
                          int32_t elem_size, int64_t b0, int64_t b1, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_fold");
    const int st = check(L, d_src_params, dst_shard, elem_size, b0, b1);
    if (st != FP8Z1_OK || b0 == b1) return st;
    return launch<true>(L, const_cast<void* const*>(d_src_params), static_cast<uint8_t*>(dst_shard),
                        elem_size, b0, b1, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8z1_unfold(const fp8z1_layout* L, const void* src_shard, void* const* d_dst_params,
                            int32_t elem_size, int64_t b0, int64_t b1, void* stream)
{
    fp8z1::NvtxRange nvtx_range("fp8z1_unfold");
    const int st = check(L, d_dst_params, src_shard, elem_size, b0, b1);
    if (st != FP8Z1_OK || b0 == b1) return st;
    return launch<false>(L, d_dst_params, const_cast<uint8_t*>(static_cast<const uint8_t*>(src_shard)),
                         elem_size, b0, b1, static_cast<cudaStream_t>(stream));
}

FP8Z1_CHECKED_MISSES_READER(checked_misses_fold)
