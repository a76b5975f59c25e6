// Internal declarations shared by the CUDA translation units of
// librope_chain.so.  Nothing here is part of the public C ABI.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "rope_chain.h"

namespace rc {

constexpr int kHidden = 8192;        // row width of the context norms
constexpr int kHeadDim = 64;         // key/value head width
constexpr int kMaxLayersPerLaunch = 8;

// ---------------------------------------------------------------- bf16

// Exact widening of the low / high bf16 of a packed pair.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round to nearest even to bf16 and back to float.
__device__ __forceinline__ float round_bf16(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

// Pack two floats, each rounded to nearest even, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// Inverse RMS of a row or head: 1 / sqrt(fma(sumsq, inv_width, eps)), each
// step correctly rounded (IEEE sqrt and divide).
__device__ __forceinline__ float inv_rms(float sumsq, float inv_width, float eps) {
    return __fdiv_rn(1.0f, __fsqrt_rn(__fmaf_rn(sumsq, inv_width, eps)));
}

// xor-butterfly sum over the 32 lanes of a warp (offsets 16, 8, 4, 2, 1).
__device__ __forceinline__ float warp_butterfly_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// The key pair (k0, k1) = elements (2 lane, 2 lane + 1) of one head, for a
// whole warp: weightless K-norm (sum folded as even and odd squares by xor
// butterflies, then even + odd), the bf16 key, GPT-J RoPE with (c, s), and
// the packed bf16 result.
template <bool kRope>
__device__ __forceinline__ uint32_t knorm_rope_lane(float k0, float k1, float c, float s, float eps) {
    const float even = warp_butterfly_sum(__fmul_rn(k0, k0));
    const float odd = warp_butterfly_sum(__fmul_rn(k1, k1));
    const float r = inv_rms(__fadd_rn(even, odd), 0x1p-6f, eps);
    float n0 = round_bf16(__fmul_rn(k0, r));
    float n1 = round_bf16(__fmul_rn(k1, r));
    if (kRope) {
        const float x = __fmaf_rn(n0, c, -__fmul_rn(n1, s));
        const float y = __fmaf_rn(n1, c, __fmul_rn(n0, s));
        n0 = x;
        n1 = y;
    }
    return pack_bf16x2(n0, n1);
}

// The head's sum over 32 pair values in the order of the lane butterfly seen
// from lane 0: (j, j+16), then partners +8, +4, +2, +1.  Every lane of the
// butterfly ends with these bits (IEEE addition commutes), so one thread
// holding the whole head reproduces the warp's sum exactly.
__device__ __forceinline__ float fold32(const float (&q)[32]) {
    float a[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        a[j] = __fadd_rn(q[j], q[j + 16]);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        a[j] = __fadd_rn(a[j], a[j + 8]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        a[j] = __fadd_rn(a[j], a[j + 4]);
#pragma unroll
    for (int j = 0; j < 2; ++j)
        a[j] = __fadd_rn(a[j], a[j + 2]);
    return __fadd_rn(a[0], a[1]);
}

// ------------------------------------------------ packed FP32 pairs
//
// The sm_100 family's .f32x2 arithmetic: one instruction works on two FP32
// values, each lane rounded to nearest once and nothing flushed to zero, so
// a lane's result has the bits of the scalar __fadd_rn / __fmul_rn /
// __fmaf_rn.

__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    unsigned long long p;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(a), "f"(b));
    return p;
}
__device__ __forceinline__ void f2_unpack(unsigned long long p, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(p));
}

// (a, b) <- (a + x, b + y)
__device__ __forceinline__ void add2_rn(float &a, float &b, float x, float y) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a, b)), "l"(f2_pack(x, y)));
    f2_unpack(r, a, b);
}
// (a, b) <- (a * x, b * y)
__device__ __forceinline__ void mul2_rn(float &a, float &b, float x, float y) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a, b)), "l"(f2_pack(x, y)));
    f2_unpack(r, a, b);
}
// (a, b) <- (fma(a, x, u), fma(b, y, v))
__device__ __forceinline__ void fma2_rn(float &a, float &b, float x, float y, float u, float v) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r) : "l"(f2_pack(a, b)), "l"(f2_pack(x, y)), "l"(f2_pack(u, v)));
    f2_unpack(r, a, b);
}

// The even and the odd square sums of a key head (w[j]: pair j = elements
// (2j, 2j+1) as packed bf16), each folded as fold32 folds: (j, j+16), then
// partners +8, +4, +2, +1.  The two trees run side by side in packed pairs.
__device__ __forceinline__ void fold32_squares2(const uint32_t (&w)[32], float &even, float &odd) {
    float e[16], o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        float x0 = bf16_lo(w[j]), x1 = bf16_hi(w[j]);
        float y0 = bf16_lo(w[j + 16]), y1 = bf16_hi(w[j + 16]);
        mul2_rn(x0, x1, x0, x1);
        mul2_rn(y0, y1, y0, y1);
        add2_rn(x0, x1, y0, y1);
        e[j] = x0;
        o[j] = x1;
    }
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
#pragma unroll
        for (int j = 0; j < s; ++j)
            add2_rn(e[j], o[j], e[j + s], o[j + s]);
    }
    even = e[0];
    odd = o[0];
}

// One key pair kw = (k0, k1) after the head's inverse RMS r: the bf16 key
// (bf16(k0 * r), bf16(k1 * r)) and with kRope the GPT-J rotation
// (fma(n0, c, -(n1 * s)), fma(n1, c, n0 * s)), packed to bf16.
template <bool kRope>
__device__ __forceinline__ uint32_t norm_rope_pair(uint32_t kw, float r, float c, float s) {
    float n0 = bf16_lo(kw), n1 = bf16_hi(kw);
    mul2_rn(n0, n1, r, r);
    const uint32_t n = pack_bf16x2(n0, n1);
    if (!kRope)
        return n;
    n0 = bf16_lo(n);
    n1 = bf16_hi(n);
    float p1 = n1, p0 = n0;                       // (n1 * s, n0 * s)
    mul2_rn(p1, p0, s, s);
    fma2_rn(n0, n1, c, c, -p1, p0);
    return pack_bf16x2(n0, n1);
}

// One whole key head in one thread: w[j] holds pair j = elements (2j, 2j+1)
// as packed bf16.  Weightless K-norm (even squares and odd squares each
// folded as fold32 does, then even + odd), the bf16 key, GPT-J RoPE with the
// table row cs (cos of pairs 0..31 in logical chunks 0..3, sin in chunks
// 4..7, 8 bf16 per 16-byte chunk; logical chunk c stored at c ^ swz), packed
// back into w.  The same operations, in the same order, as knorm_rope_lane.
template <bool kRope>
__device__ __forceinline__ void knorm_rope_head(uint32_t (&w)[32], const uint4 *cs, int swz,
                                                float eps) {
    float even, odd;
    fold32_squares2(w, even, odd);
    const float r = inv_rms(__fadd_rn(even, odd), 0x1p-6f, eps);
#pragma unroll
    for (int q = 0; q < 4; ++q) {                 // 8 pairs per table chunk
        uint4 c4 = make_uint4(0, 0, 0, 0), s4 = c4;
        if (kRope) {
            c4 = cs[q ^ swz];
            s4 = cs[(4 + q) ^ swz];
        }
        const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w}, sw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int j = 8 * q + t;
            const float c = (t & 1) ? bf16_hi(cw[t >> 1]) : bf16_lo(cw[t >> 1]);
            const float s = (t & 1) ? bf16_hi(sw[t >> 1]) : bf16_lo(sw[t >> 1]);
            w[j] = norm_rope_pair<kRope>(w[j], r, c, s);
        }
    }
}

// ------------------------------------------------- programmatic launches
//
// Every kernel of the library is launched with programmatic stream
// serialization: it may start while the previous kernel on the stream is
// finishing.  Each kernel lets its own dependents launch as soon as it starts
// (pdl_trigger) and touches no global memory before pdl_wait, which returns
// once the previous kernel has completed and its writes are visible; so only
// launch latency and prologue work (barrier set-up, TMEM allocation) overlap.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// cudaLaunchKernelEx with programmatic stream serialization and, when
// cluster_x > 1, a (cluster_x, 1, 1) cluster.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned n = 1;
    if (cluster_x > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------- launches

// Norms: grid of T CTAs x 256 threads (T / 2 with two rows per CTA);
// returns the launch error.  bf16 output-scale weights (or none), gain
// center 0.  `early`: the kernel does not wait for the kernel before it in
// the stream (the caller guarantees that kernel neither reads out nor writes
// x or the weights), and its last CTA waits for it before exiting.
cudaError_t launch_context_norms(const uint16_t *x, int64_t T, const uint16_t *hidden_w,
                                 const uint16_t *pre_w, int32_t L, float hidden_eps, float pre_eps,
                                 uint16_t *out, cudaStream_t stream, bool early = false);

// One norm of the variant kernel: weight NULL (weightless), bf16 or FP32
// ([8192] hidden, [L, 8192] layers), whether it scales the input, its gain
// center (added when non-zero) and eps.
struct NormDesc {
    const void *w;
    int32_t fp32;
    int32_t input_scale;
    float center;
    float eps;
};

cudaError_t launch_context_norms_ex(const uint16_t *x, int64_t T, const NormDesc &hidden,
                                    const NormDesc &pre, int32_t L, uint16_t *out,
                                    cudaStream_t stream, bool early = false);

// Row prep for the fused chain: z = bf16 [T, 8192] hidden-norm output and
// r2 [T] = the layers' shared inverse RMS of z.
cudaError_t launch_row_prep(const uint16_t *x, int64_t T, const uint16_t *hidden_w, float eps,
                            uint16_t *z, float *r2, cudaStream_t stream);

struct StoreLaunch {
    const uint16_t *k;               // layer 0 of this chunk
    const uint16_t *v;
    int64_t k_layer_stride, k_row_stride, v_layer_stride, v_row_stride;   // elements
    const int64_t *positions;
    const uint16_t *cos_sin;
    int64_t max_position;
    const int64_t *slots[kMaxLayersPerLaunch];
    uint16_t *caches[kMaxLayersPerLaunch];
    int64_t capacity;                // num_blocks * block_size
    int32_t block_size;
    int32_t rows[kMaxLayersPerLaunch];   // rows inserted per layer of the chunk
    int32_t grid_rows;               // rows the grid covers (max over the chunk)
    float eps;
    int32_t *err;
};

// The store half of the fused projection + store (all layers in one launch).
constexpr int kMaxFusedLayers = 64;
struct FusedStore {
    const int64_t *positions;
    const uint16_t *cos_sin;         // NULL: no RoPE
    int64_t max_position;
    const int64_t *slots[kMaxFusedLayers];
    uint16_t *caches[kMaxFusedLayers];
    int64_t capacity;                // num_blocks * block_size
    int32_t block_size;
    int32_t H;
    int32_t rows[kMaxFusedLayers];   // rows inserted per layer (<= T)
    float eps;
    int32_t *err;
    uint16_t *kv_out;                // optional bf16 [L, T, 2*H*64] copy of the projection
};

// Store from split-K partials: adds the FP32 partials [splits, L, T, N] in
// split order, rounds to bf16 (the projection), then K-norm, RoPE and insert.
cudaError_t launch_reduce_store(const FusedStore &fs, const float *partial, int32_t splits,
                                int32_t L, int32_t T, cudaStream_t stream);

// Store: one chunk of <= 8 layers; H in {1,2,4,8,16,32}.
cudaError_t launch_kv_store(const StoreLaunch &p, int32_t H, int32_t layers,
                            cudaStream_t stream);

struct ProjectPlan {
    bool pair;             // CTA pairs (cta_group::2, 256 x 256 tiles)
    int bn;                // 128 or 256
    int splits;            // >= 1
    int kb_per_split;      // 64-wide K blocks per split
    // Persistent pair plans whose last wave would leave most pairs idle:
    // the last tail_tiles tiles (rows tail_row0 .. T-1 of the last layer)
    // run as their own split-K launch (tail_splits splits of
    // tail_kb_per_split K blocks) after the persistent kernel's full waves.
    int64_t tail_tiles;    // 0: no tail launch
    int64_t tail_row0;
    int tail_splits;
    int tail_kb_per_split;
    // Persistent pair plans of eight rounds of tiles or more: byte offset in
    // the workspace of the 4-byte counter (zeroed by the call) from which
    // the pairs take tiles in order (dynamic tile order); -1: each pair takes
    // a fixed sequence.
    int64_t tile_ctr_offset;
    size_t workspace;      // bytes used: FP32 partials (split-K or the tail's), then the counter
    // The caller zeroed the tile counter earlier in the stream (no memset
    // between the kernel before and the projection).
    bool ctr_zeroed;
};

// Choose tile width and split count for the device's SM count.  Without
// allow_tail no tail launch is planned (the forming projection of the whole
// chain takes every tile itself).
ProjectPlan plan_kv_project(int32_t L, int64_t T, int32_t D, int32_t N, int num_sms,
                            size_t workspace_bytes, bool allow_tail = true);

// Projection; `ws` holds the FP32 partials when plan.splits > 1.
cudaError_t launch_kv_project(const uint16_t *normed, const uint16_t *W, bool w_nk,
                              uint16_t *out, int32_t L, int64_t T, int32_t D, int32_t N,
                              const ProjectPlan &plan, float *ws, cudaStream_t stream,
                              const char **why);

// Sets the message rc_last_error() returns on this host thread.
void set_last_error(const char *msg);

// The argument checks of rc_kv_project (sizes, weight layout, NULL and
// 16-byte alignment of normed, W and out, out overlapping an input); on a
// refusal the message names `fn` and the status is returned.
rc_status check_project_call(const char *fn, const uint16_t *normed, const uint16_t *W,
                             int32_t w_layout, const uint16_t *out, int32_t L, int64_t T,
                             int32_t D, int32_t N);

// Projection + store: the pair kernel's epilogue stores when it does not
// split; split plans go through launch_reduce_store; single-CTA plans that do
// not split need fs.kv_out (projection to kv_out, then the store kernel).
cudaError_t launch_kv_project_store(const uint16_t *normed, const uint16_t *W, bool w_nk,
                                    int32_t L, int64_t T, int32_t D, int32_t N,
                                    const ProjectPlan &plan, float *ws, const FusedStore &fs,
                                    cudaStream_t stream, const char **why);

// The chain after the row pass, for CTA-pair plans: the projection forming
// each layer's normed tile from (z, r2, pre_w) in shared memory, with the
// store fused (epilogue, or the reduce-and-store pass when K is split).
cudaError_t launch_kv_from_rows(const uint16_t *z, const float *r2, int64_t T,
                                const uint16_t *pre_w, const uint16_t *W, bool w_nk, int32_t L,
                                int32_t N, const ProjectPlan &plan, float *ws, const FusedStore &fs,
                                cudaStream_t stream, const char **why);

// Sticky device fault bits of the projection kernel (current device).
cudaError_t read_project_faults(uint32_t *flags, bool clear);

// The decode QKV front (1 to 16 tokens): projection, QK-norm, RoPE, insert.
cudaError_t launch_qkv_front(const uint16_t *hidden, int32_t M, int32_t D, const uint16_t *W,
                             int32_t num_heads, int32_t num_kv_heads, const int64_t *positions,
                             const uint16_t *cos_sin, int64_t max_position, const int64_t *slots,
                             uint16_t *cache, int32_t num_blocks, int32_t block_size, float eps,
                             uint16_t *out, uint16_t *raw, int32_t *err, int num_sms,
                             cudaStream_t stream, const char **why);

// Sticky device fault bits of the QKV front kernel (current device).
cudaError_t read_front_faults(uint32_t *flags, bool clear);

}  // namespace rc
