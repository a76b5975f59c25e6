// K3: K-norm, GPT-J RoPE and the paged insert of K and V.
//
// Page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context",
// _ContextKvStoreKernel / _sum_squares_64 / _rope: one warp per (row, layer),
// lane j holding the GPT-J pair (2j, 2j+1) of every head, the head's sum of
// squares folded as even squares and odd squares separately by an xor
// butterfly, then even + odd; the normed key rounded to bf16; the rotation
// (fma(x, c, -(y*s)), fma(y, c, x*s)); K and V written as 4-byte words, so
// each warp store covers 128 contiguous bytes of one head.
//
// Differences from the pages' kernel: 8 warps (rows) per CTA instead of one;
// a slot past the cache or a position past the table skips the row and counts
// it in the caller's error word instead of writing out of bounds.
#include "rc_internal.cuh"

namespace rc {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void count_skip(int32_t *err, int lane) {
    if (err != nullptr && lane == 0)
        atomicAdd(err, 1);
}

// Writes one row's H heads of K' and V into its cache slot (lane = pair).
template <int H>
__device__ __forceinline__ void insert_row(uint16_t *cache, int64_t slot, int32_t block_size,
                                           const uint32_t (&ko)[H], const uint32_t (&vw)[H],
                                           int lane) {
    // Slots of a cache fit 32 bits (checked on the host).
    const uint32_t bs = (uint32_t)block_size;
    const uint32_t blk = (uint32_t)slot / bs;
    const uint32_t page = (uint32_t)slot - blk * bs;
    uint32_t *dst = reinterpret_cast<uint32_t *>(cache) + (((int64_t)blk * H) * bs + page) * kHeadDim + lane;
    const int64_t head_stride = (int64_t)bs * kHeadDim;      // in 4-byte words
#pragma unroll
    for (int h = 0; h < H; ++h) {
        dst[h * head_stride] = ko[h];
        dst[h * head_stride + kHeadDim / 2] = vw[h];          // V follows K
    }
}

template <int H, bool kRope>
__global__ void __launch_bounds__(kWarps * 32)
k3_kv_store(const __grid_constant__ StoreLaunch p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    const int layer = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    if (row >= p.rows[layer])
        return;
    const int64_t *slots = p.slots[layer];
    if (slots == nullptr)
        return;
    // Every load first, as the pages' kernel does: the slot, the position and
    // the row's K and V words are independent, so their latencies overlap; a
    // skipped row wastes its K/V reads but never writes.
    const int64_t slot = __ldg(slots + row);
    const int64_t pos = kRope ? __ldg(p.positions + row) : 0;
    const uint32_t *kr = reinterpret_cast<const uint32_t *>(
        p.k + (int64_t)layer * p.k_layer_stride + row * p.k_row_stride) + lane;
    const uint32_t *vr = reinterpret_cast<const uint32_t *>(
        p.v + (int64_t)layer * p.v_layer_stride + row * p.v_row_stride) + lane;
    uint32_t kw[H], vw[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        kw[h] = __ldcs(kr + h * (kHeadDim / 2));
        vw[h] = __ldcs(vr + h * (kHeadDim / 2));
    }
    if (slot < 0)
        return;
    if (slot >= p.capacity || (kRope && (pos < 0 || pos >= p.max_position))) {
        count_skip(p.err, lane);
        return;
    }
    float c = 1.0f, s = 0.0f;
    if (kRope) {
        const unsigned short *cs = reinterpret_cast<const unsigned short *>(p.cos_sin) + pos * kHeadDim;
        c = __uint_as_float((uint32_t)__ldg(cs + lane) << 16);
        s = __uint_as_float((uint32_t)__ldg(cs + kHeadDim / 2 + lane) << 16);
    }

    uint32_t ko[H];
#pragma unroll
    for (int h = 0; h < H; ++h)
        ko[h] = knorm_rope_lane<kRope>(bf16_lo(kw[h]), bf16_hi(kw[h]), c, s, p.eps);
    insert_row<H>(p.caches[layer], slot, p.block_size, ko, vw, lane);
}

// Split-K projection finished and stored in one pass: the FP32 partials
// [splits, L, T, 128 H] are added in split order and rounded to bf16 (the
// same additions as the projection's reduce kernel), optionally written to
// kv_out, and stored like k3_kv_store.  One warp per (row, layer, head): the
// K-norm needs only its head, and many splits (small T) still leave enough
// warps; the split loop is unrolled so 8 partials are in flight per lane.
template <bool kRope>
__global__ void __launch_bounds__(kWarps * 32)
k3_reduce_store(const __grid_constant__ FusedStore fs, const float *__restrict__ partial,
                int32_t splits, int32_t L, int32_t T)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    const int layer = blockIdx.y;
    const int h = blockIdx.z;
    const int H = fs.H;
    const int N = 2 * H * kHeadDim;
    pdl_trigger();
    pdl_wait();
    if (row >= T)
        return;
    const int64_t *slots = fs.slots[layer];
    const bool store = slots != nullptr && row < fs.rows[layer];
    int64_t slot = -1, pos = 0;
    if (store) {
        slot = __ldg(slots + row);
        if (kRope)
            pos = __ldg(fs.positions + row);
    }
    const int64_t plane = (int64_t)L * T * N;
    const float *pk = partial + ((int64_t)layer * T + row) * N + h * kHeadDim + 2 * lane;
    const float *pv = pk + H * kHeadDim;
    float2 ka = __ldcs(reinterpret_cast<const float2 *>(pk));
    float2 va = __ldcs(reinterpret_cast<const float2 *>(pv));
    int sp = 1;
    for (; sp + 8 <= splits; sp += 8) {
        float2 a[8], b[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            a[u] = __ldcs(reinterpret_cast<const float2 *>(pk + (sp + u) * plane));
            b[u] = __ldcs(reinterpret_cast<const float2 *>(pv + (sp + u) * plane));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            ka.x = __fadd_rn(ka.x, a[u].x);
            ka.y = __fadd_rn(ka.y, a[u].y);
            va.x = __fadd_rn(va.x, b[u].x);
            va.y = __fadd_rn(va.y, b[u].y);
        }
    }
    for (; sp < splits; ++sp) {
        const float2 a = __ldcs(reinterpret_cast<const float2 *>(pk + sp * plane));
        const float2 b = __ldcs(reinterpret_cast<const float2 *>(pv + sp * plane));
        ka.x = __fadd_rn(ka.x, a.x);
        ka.y = __fadd_rn(ka.y, a.y);
        va.x = __fadd_rn(va.x, b.x);
        va.y = __fadd_rn(va.y, b.y);
    }
    const uint32_t kw = pack_bf16x2(ka.x, ka.y), vw = pack_bf16x2(va.x, va.y);
    if (fs.kv_out != nullptr) {
        uint32_t *o = reinterpret_cast<uint32_t *>(fs.kv_out + ((int64_t)layer * T + row) * N) + lane;
        o[h * (kHeadDim / 2)] = kw;
        o[(H + h) * (kHeadDim / 2)] = vw;
    }
    if (!store || slot < 0)
        return;
    if (slot >= fs.capacity || (kRope && (pos < 0 || pos >= fs.max_position))) {
        if (h == 0)                               // once per (row, layer)
            count_skip(fs.err, lane);
        return;
    }
    float c = 1.0f, s = 0.0f;
    if (kRope) {
        const unsigned short *cs = reinterpret_cast<const unsigned short *>(fs.cos_sin) + pos * kHeadDim;
        c = __uint_as_float((uint32_t)__ldg(cs + lane) << 16);
        s = __uint_as_float((uint32_t)__ldg(cs + kHeadDim / 2 + lane) << 16);
    }
    const uint32_t ko = knorm_rope_lane<kRope>(bf16_lo(kw), bf16_hi(kw), c, s, fs.eps);
    // Slots of a cache fit 32 bits (checked on the host).
    const uint32_t bs = (uint32_t)fs.block_size;
    const uint32_t blk = (uint32_t)slot / bs;
    const uint32_t page = (uint32_t)slot - blk * bs;
    uint32_t *dst = reinterpret_cast<uint32_t *>(fs.caches[layer]) +
                    (((int64_t)blk * H + h) * bs + page) * kHeadDim + lane;
    dst[0] = ko;
    dst[kHeadDim / 2] = vw;                       // V follows K
}

template <int H>
cudaError_t launch_h(const StoreLaunch &p, int32_t layers, cudaStream_t stream) {
    const dim3 grid((unsigned)((p.grid_rows + kWarps - 1) / kWarps), (unsigned)layers);
    if (p.cos_sin)
        return launch_pdl(k3_kv_store<H, true>, grid, dim3(kWarps * 32), 0, stream, 1, p);
    return launch_pdl(k3_kv_store<H, false>, grid, dim3(kWarps * 32), 0, stream, 1, p);
}

}  // namespace

cudaError_t launch_reduce_store(const FusedStore &fs, const float *partial, int32_t splits,
                                int32_t L, int32_t T, cudaStream_t stream)
{
    const dim3 grid((unsigned)((T + kWarps - 1) / kWarps), (unsigned)L, (unsigned)fs.H);
    if (fs.cos_sin)
        return launch_pdl(k3_reduce_store<true>, grid, dim3(kWarps * 32), 0, stream, 1, fs, partial,
                          splits, L, T);
    return launch_pdl(k3_reduce_store<false>, grid, dim3(kWarps * 32), 0, stream, 1, fs, partial,
                      splits, L, T);
}

cudaError_t launch_kv_store(const StoreLaunch &p, int32_t H, int32_t layers, cudaStream_t stream)
{
    switch (H) {
    case 1: return launch_h<1>(p, layers, stream);
    case 2: return launch_h<2>(p, layers, stream);
    case 4: return launch_h<4>(p, layers, stream);
    case 8: return launch_h<8>(p, layers, stream);
    case 16: return launch_h<16>(p, layers, stream);
    case 32: return launch_h<32>(p, layers, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rc
