// K1: the context norms (hidden RMSNorm -> bf16 -> each layer's input
// RMSNorm, stacked to [L, T, 8192]).
//
// Page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context",
// _ContextNormsKernel: 256 threads per row, thread t holding the 16-byte
// fragments at columns 8t + 2048k (k < 4), the hidden norm's output rounded
// to bf16 before the layer norm reads it.  The pages launch one CTA per
// (row, layer) and recompute the hidden norm L times; here one CTA handles a
// row for all L layers: x is read once, both row sums are taken once (the
// layer gains scale the norm's output, so the layer norm's inverse RMS is
// the same for every layer), and only the per-layer scale and store repeat.
//
// Order of the sums (fixed, and the oracle's reading R1): each thread adds
// its 32 squares in (k, i) order, each warp folds its 32 partials with an xor
// butterfly, and the 8 warp sums are added left to right by every thread.
#include "rc_internal.cuh"

namespace rc {
namespace {

constexpr int kThreads = 256;
constexpr int kFrags = 4;             // 16-byte fragments per thread
constexpr int kFragStride = 256;      // uint4 units between a thread's fragments
constexpr int64_t kTwoRowsFrom = 16384;   // rows from which a CTA takes two
constexpr int64_t kExTwoRowsFrom = 16384; // the same for the norm-options kernel (weights staged)

__device__ __forceinline__ void unpack8(const uint4 &q, float *f) {
    f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x);
    f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
    f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z);
    f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
}

// Sum of squares of the row this CTA holds (its 4 packed fragments per
// thread), in the documented order.
__device__ __forceinline__ float row_sumsq(const uint4 (&q)[kFrags], float *sums, int warp,
                                           int lane) {
    float p = 0.0f;
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        float f[8];
        unpack8(q[k], f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p = __fadd_rn(p, __fmul_rn(f[i], f[i]));
    }
    p = warp_butterfly_sum(p);
    if (lane == 0)
        sums[warp] = p;
    __syncthreads();
    float s = sums[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w)
        s = __fadd_rn(s, sums[w]);
    return s;
}

__device__ __forceinline__ uint4 pack8(const float *y) {
    uint4 w;
    w.x = pack_bf16x2(y[0], y[1]);
    w.y = pack_bf16x2(y[2], y[3]);
    w.z = pack_bf16x2(y[4], y[5]);
    w.w = pack_bf16x2(y[6], y[7]);
    return w;
}

// `early`: the kernel was launched while the kernel before it in the stream
// still runs, and touches nothing that kernel reads or writes, so it does not
// wait for it at the start.  It still completes after it: its last CTA waits
// for that kernel before exiting, so a kernel that waits for this one (the
// projection of these rows) has also waited for the one before.
__device__ __forceinline__ void early_join(int early) {
    if (early && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
        pdl_wait();
}

template <bool kHiddenW, bool kPreW>
__global__ void __launch_bounds__(kThreads, 4)
k1_context_norms(const uint16_t *__restrict__ x, int64_t T,
                 const uint16_t *__restrict__ hidden_w, const uint16_t *__restrict__ pre_w,
                 int32_t L, float hidden_eps, float pre_eps, uint16_t *__restrict__ out,
                 int early)
{
    __shared__ float sums[2][kThreads / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row = blockIdx.x;
    pdl_trigger();
    if (!early)
        pdl_wait();

    // The row (read once: streaming) and the hidden gains (shared by all
    // rows: cached) load together.
    const uint4 *xr = reinterpret_cast<const uint4 *>(x) + row * (kHidden / 8);
    const uint4 *gh = reinterpret_cast<const uint4 *>(hidden_w);
    const uint4 *gp = reinterpret_cast<const uint4 *>(pre_w);
    uint4 q[kFrags], hq[kFrags], pq[kFrags];
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        q[k] = __ldcs(xr + k * kFragStride + tid);
        if (kHiddenW)
            hq[k] = __ldg(gh + k * kFragStride + tid);
    }

    // a1: hidden norm; z = bf16((x * r) * gamma) kept packed in q
    const float r = inv_rms(row_sumsq(q, sums[0], warp, lane), 0x1p-13f, hidden_eps);
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        float f[8];
        unpack8(q[k], f);
        if (kHiddenW) {
            float g[8];
            unpack8(hq[k], g);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = __fmul_rn(__fmul_rn(f[i], r), g[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = __fmul_rn(f[i], r);
        }
        q[k] = pack8(f);
    }

    // Layer 0's gains load while the second row sum is reduced.
    if (kPreW) {
#pragma unroll
        for (int k = 0; k < kFrags; ++k)
            pq[k] = __ldg(gp + k * kFragStride + tid);
    }

    // a2: the layers' input norms share one inverse RMS
    const float r2 = inv_rms(row_sumsq(q, sums[1], warp, lane), 0x1p-13f, pre_eps);
    for (int32_t l = 0; l < L; ++l) {
        uint4 *o = reinterpret_cast<uint4 *>(out) + ((int64_t)l * T + row) * (kHidden / 8);
        const uint4 *gn = gp + (int64_t)(l + 1) * (kHidden / 8);
#pragma unroll
        for (int k = 0; k < kFrags; ++k) {
            float f[8];
            unpack8(q[k], f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = __fmul_rn(f[i], r2);
            if (kPreW) {
                float g[8];
                unpack8(pq[k], g);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    f[i] = __fmul_rn(f[i], g[i]);
                if (l + 1 < L)                   // this fragment's gains for the next layer
                    pq[k] = __ldg(gn + k * kFragStride + tid);
            }
            o[k * kFragStride + tid] = pack8(f);
        }
    }
    early_join(early);
}

// The same norms with two rows per CTA: each thread holds its 32 columns of
// both rows, so every gain fragment is read once for the two rows (half the
// gain traffic), and each row's sums keep row_sumsq's order.  Used when
// there are enough rows to fill the GPU with half as many CTAs.
template <bool kHiddenW, bool kPreW>
__global__ void __launch_bounds__(kThreads, 2)
k1_context_norms2(const uint16_t *__restrict__ x, int64_t T,
                  const uint16_t *__restrict__ hidden_w, const uint16_t *__restrict__ pre_w,
                  int32_t L, float hidden_eps, float pre_eps, uint16_t *__restrict__ out,
                  int early)
{
    __shared__ float sums[2][2][kThreads / 32];    // [norm][row of the pair][warp]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row0 = 2 * (int64_t)blockIdx.x;
    const bool two = row0 + 1 < T;
    pdl_trigger();
    if (!early)
        pdl_wait();

    const uint4 *xa = reinterpret_cast<const uint4 *>(x) + row0 * (kHidden / 8);
    const uint4 *xb = xa + kHidden / 8;
    const uint4 *gh = reinterpret_cast<const uint4 *>(hidden_w);
    const uint4 *gp = reinterpret_cast<const uint4 *>(pre_w);
    uint4 a[kFrags], b[kFrags], hq[kFrags], pq[kFrags];
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        a[k] = __ldcs(xa + k * kFragStride + tid);
        b[k] = two ? __ldcs(xb + k * kFragStride + tid) : make_uint4(0, 0, 0, 0);
        if (kHiddenW)
            hq[k] = __ldg(gh + k * kFragStride + tid);
    }

    // one norm's inverse RMS for both rows, each in row_sumsq's order
    auto pair_scale = [&](float (&sbuf)[2][kThreads / 32], float eps, float &ra, float &rb) {
        float pa = 0.0f, pb = 0.0f;
#pragma unroll
        for (int k = 0; k < kFrags; ++k) {
            float fa[8], fb[8];
            unpack8(a[k], fa);
            unpack8(b[k], fb);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pa = __fadd_rn(pa, __fmul_rn(fa[i], fa[i]));
                pb = __fadd_rn(pb, __fmul_rn(fb[i], fb[i]));
            }
        }
        pa = warp_butterfly_sum(pa);
        pb = warp_butterfly_sum(pb);
        if (lane == 0) {
            sbuf[0][warp] = pa;
            sbuf[1][warp] = pb;
        }
        __syncthreads();
        float sa = sbuf[0][0], sb = sbuf[1][0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) {
            sa = __fadd_rn(sa, sbuf[0][w]);
            sb = __fadd_rn(sb, sbuf[1][w]);
        }
        ra = inv_rms(sa, 0x1p-13f, eps);
        rb = inv_rms(sb, 0x1p-13f, eps);
    };

    // a1: hidden norm; z = bf16((x * r) * gamma) kept packed in a and b
    float ra, rb;
    pair_scale(sums[0], hidden_eps, ra, rb);
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        float fa[8], fb[8];
        unpack8(a[k], fa);
        unpack8(b[k], fb);
        if (kHiddenW) {
            float g[8];
            unpack8(hq[k], g);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                fa[i] = __fmul_rn(__fmul_rn(fa[i], ra), g[i]);
                fb[i] = __fmul_rn(__fmul_rn(fb[i], rb), g[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                fa[i] = __fmul_rn(fa[i], ra);
                fb[i] = __fmul_rn(fb[i], rb);
            }
        }
        a[k] = pack8(fa);
        b[k] = pack8(fb);
    }
    if (kPreW) {
#pragma unroll
        for (int k = 0; k < kFrags; ++k)
            pq[k] = __ldg(gp + k * kFragStride + tid);
    }

    // a2: the layers' input norms share one inverse RMS per row
    float r2a, r2b;
    pair_scale(sums[1], pre_eps, r2a, r2b);
    for (int32_t l = 0; l < L; ++l) {
        uint4 *oa = reinterpret_cast<uint4 *>(out) + ((int64_t)l * T + row0) * (kHidden / 8);
        uint4 *ob = oa + kHidden / 8;
        const uint4 *gn = gp + (int64_t)(l + 1) * (kHidden / 8);
#pragma unroll
        for (int k = 0; k < kFrags; ++k) {
            float fa[8], fb[8];
            unpack8(a[k], fa);
            unpack8(b[k], fb);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                fa[i] = __fmul_rn(fa[i], r2a);
                fb[i] = __fmul_rn(fb[i], r2b);
            }
            if (kPreW) {
                float g[8];
                unpack8(pq[k], g);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    fa[i] = __fmul_rn(fa[i], g[i]);
                    fb[i] = __fmul_rn(fb[i], g[i]);
                }
                if (l + 1 < L)                   // this fragment's gains for the next layer
                    pq[k] = __ldg(gn + k * kFragStride + tid);
            }
            oa[k * kFragStride + tid] = pack8(fa);
            if (two)
                ob[k * kFragStride + tid] = pack8(fb);
        }
    }
    early_join(early);
}

// The row half of the norms for the fused chain: z = bf16(hidden_norm(x))
// and r2 = the layers' shared inverse RMS of z, per row; the projection
// forms each layer's bf16((z * r2) * gamma_l) tile itself.  Same arithmetic
// and order as k1_context_norms.
template <bool kHiddenW>
__global__ void __launch_bounds__(kThreads, 4)
k1_row_prep(const uint16_t *__restrict__ x, const uint16_t *__restrict__ hidden_w, float eps,
            uint16_t *__restrict__ z, float *__restrict__ r2_out)
{
    __shared__ float sums[2][kThreads / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    const uint4 *xr = reinterpret_cast<const uint4 *>(x) + row * (kHidden / 8);
    const uint4 *gh = reinterpret_cast<const uint4 *>(hidden_w);
    uint4 q[kFrags], hq[kFrags];
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        q[k] = __ldcs(xr + k * kFragStride + tid);
        if (kHiddenW)
            hq[k] = __ldg(gh + k * kFragStride + tid);
    }
    const float r = inv_rms(row_sumsq(q, sums[0], warp, lane), 0x1p-13f, eps);
    uint4 *zr = reinterpret_cast<uint4 *>(z) + row * (kHidden / 8);
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        float f[8];
        unpack8(q[k], f);
        if (kHiddenW) {
            float g[8];
            unpack8(hq[k], g);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = __fmul_rn(__fmul_rn(f[i], r), g[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = __fmul_rn(f[i], r);
        }
        q[k] = pack8(f);
        zr[k * kFragStride + tid] = q[k];
    }
    const float r2 = inv_rms(row_sumsq(q, sums[1], warp, lane), 0x1p-13f, eps);
    if (tid == 0)
        r2_out[row] = r2;
}

// ------------------------------------------------------------ variants
//
// Every option of the pages' ContextNormConstants and ContextNorms: each
// norm's weight may be absent, bf16 or FP32, may scale the norm's input
// (before the sum of squares) or its output, has a gain center added to
// each element when non-zero, and its own eps.  With an input-scale layer
// weight the layers' inverse RMS differs per layer, so each layer takes its
// own row sum.  Same thread mapping, order of sums and roundings as
// k1_context_norms; the options are uniform over the grid, so the branches
// on them do not diverge.

// Fragment k's 8 gains of weight row `row` (its columns 2048 k + 8 t + i).
__device__ __forceinline__ void load_gains(const NormDesc &n, int64_t row, int k, int tid,
                                           float (&g)[8]) {
    const int64_t col = row * kHidden + (int64_t)k * 2048 + 8 * tid;
    if (n.fp32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(n.w) + col);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
        g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
    } else {
        unpack8(__ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(n.w) + col)), g);
    }
    if (n.center != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            g[i] = __fadd_rn(g[i], n.center);
    }
}

// Inverse RMS of one norm of R rows held packed in q (row j in q[j]): the
// sum of squares of each row's inputs (the packed bf16 values, times the
// gains when the weight scales the input) in the order of row_sumsq -- each
// thread's 32 values in (k, i) order, an xor butterfly per warp, the 8 warp
// sums left to right -- then 1 / sqrt(fma(S, 2^-13, eps)).  Each gain
// fragment is loaded once for the R rows.  `sums` alternates between two
// buffers so that consecutive norms need one barrier each.
template <int R>
__device__ __forceinline__ void norm_scale(const uint4 (&q)[R][kFrags], const NormDesc &n,
                                           int64_t wrow, float (&sums)[2][R][kThreads / 32],
                                           int &buf, int tid, int warp, int lane, float (&r)[R]) {
    const bool in_scale = n.w != nullptr && n.input_scale;
    float p[R];
#pragma unroll
    for (int j = 0; j < R; ++j)
        p[j] = 0.0f;
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        float g[8];
        if (in_scale)
            load_gains(n, wrow, k, tid, g);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float f[8];
            unpack8(q[j][k], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (in_scale)
                    f[i] = __fmul_rn(g[i], f[i]);
                p[j] = __fadd_rn(p[j], __fmul_rn(f[i], f[i]));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
        p[j] = warp_butterfly_sum(p[j]);
        if (lane == 0)
            sums[buf][j][warp] = p[j];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < R; ++j) {
        float s = sums[buf][j][0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w)
            s = __fadd_rn(s, sums[buf][j][w]);
        r[j] = inv_rms(s, 0x1p-13f, n.eps);
    }
    buf ^= 1;
}

// Fragment k of one norm's output for R rows: (input * r), times the gains
// when the weight scales the output, packed to bf16 (the gain fragment read
// once for the R rows).
template <int R>
__device__ __forceinline__ void norm_output(const uint4 (&q)[R][kFrags], const NormDesc &n,
                                            int64_t wrow, int k, int tid, const float (&r)[R],
                                            uint4 (&o)[R]) {
    const bool weighted = n.w != nullptr;
    float g[8];
    if (weighted)
        load_gains(n, wrow, k, tid, g);
#pragma unroll
    for (int j = 0; j < R; ++j) {
        float f[8];
        unpack8(q[j][k], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (weighted && n.input_scale)
                f[i] = __fmul_rn(g[i], f[i]);
            f[i] = __fmul_rn(f[i], r[j]);
            if (weighted && !n.input_scale)
                f[i] = __fmul_rn(f[i], g[i]);
        }
        o[j] = pack8(f);
    }
}

// Both norms with every option: each weight bf16, FP32 or absent, scaling
// the norm's input (gamma * x, before the sum of squares) or its output,
// a gain center added when non-zero, its own eps.  With an input-scale
// layer weight the layers' inverse RMS differs per layer, so each layer
// takes its own row sum.  Same thread mapping, order of sums and roundings
// as k1_context_norms; R rows per CTA (run with one; the helpers take R for
// the staged kernel below); the rows stay packed and each fragment is formed
// on its own (few live registers); the options are uniform over the grid,
// so the branches on them do not diverge.
template <int R>
__global__ void __launch_bounds__(kThreads, 4)
k1_context_norms_ex(const uint16_t *__restrict__ x, int64_t T, const NormDesc hidden,
                    const NormDesc pre, int32_t L, uint16_t *__restrict__ out, int early)
{
    __shared__ float sums[2][R][kThreads / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row0 = (int64_t)blockIdx.x * R;
    int buf = 0;
    pdl_trigger();
    if (!early)
        pdl_wait();

    uint4 q[R][kFrags];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const bool live = row0 + j < T;             // a missing last row reads as zeros
        const uint4 *xr = reinterpret_cast<const uint4 *>(x) + (row0 + j) * (kHidden / 8);
#pragma unroll
        for (int k = 0; k < kFrags; ++k)
            q[j][k] = live ? __ldcs(xr + k * kFragStride + tid) : make_uint4(0, 0, 0, 0);
    }
    // a1: the hidden norm, rounded to bf16 (z kept packed)
    float r[R];
    norm_scale<R>(q, hidden, 0, sums, buf, tid, warp, lane, r);
    uint4 z[R][kFrags];
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        uint4 o[R];
        norm_output<R>(q, hidden, 0, k, tid, r, o);
#pragma unroll
        for (int j = 0; j < R; ++j)
            z[j][k] = o[j];
    }

    // a2: with an output-scale (or no) layer weight one inverse RMS serves
    // every layer
    const bool per_layer = pre.w != nullptr && pre.input_scale;
    float r2[R];
    if (!per_layer) {
        NormDesc plain = pre;
        plain.w = nullptr;                       // the sum is of z itself
        norm_scale<R>(z, plain, 0, sums, buf, tid, warp, lane, r2);
    }
    // each layer's fragment gains read where they are used (this keeps the
    // registers, and so the occupancy, of the plain kernel)
    for (int32_t l = 0; l < L; ++l) {
        float rl[R];
        if (per_layer) {
            norm_scale<R>(z, pre, l, sums, buf, tid, warp, lane, rl);
        } else {
#pragma unroll
            for (int j = 0; j < R; ++j)
                rl[j] = r2[j];
        }
#pragma unroll
        for (int k = 0; k < kFrags; ++k) {
            uint4 o[R];
            norm_output<R>(z, pre, l, k, tid, rl, o);
#pragma unroll
            for (int j = 0; j < R; ++j)
                if (row0 + j < T)
                    reinterpret_cast<uint4 *>(out)[((int64_t)l * T + row0 + j) * (kHidden / 8) +
                                                   k * kFragStride + tid] = o[j];
        }
    }
    early_join(early);
}

// ---- the same kernel with each weight row staged in shared memory
//
// With FP32 gains a layer's weight row is 32 KiB, and L of them do not stay
// in L1, so reading each fragment's gains from global memory once per CTA
// costs as much L2 traffic as the rows themselves.  Here the CTA copies each
// weight row into shared memory once (cp.async, two buffers: the next
// layer's row lands while this layer is stored) and R rows share it; no gain
// is held in registers across the layer loop.  Same arithmetic and order.

constexpr int kGainBytes = kHidden * 4;          // one FP32 weight row

// Start copying weight row `row` of n into dst (a no-op without a weight);
// always commits one group, so the group count is the same for every option.
__device__ __forceinline__ void stage_gains(const NormDesc &n, int64_t row, uint8_t *dst, int tid) {
    if (n.w != nullptr) {
        const int bytes = n.fp32 ? kHidden * 4 : kHidden * 2;
        const uint8_t *src = static_cast<const uint8_t *>(n.w) + row * bytes;
        for (int o = 16 * tid; o < bytes; o += 16 * kThreads) {
            const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst + o));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src + o) : "memory");
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void staged_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Fragment k's 8 gains (columns 2048 k + 8 t + i) from a staged weight row.
__device__ __forceinline__ void smem_gains(const NormDesc &n, const uint8_t *row, int k, int tid,
                                           float (&g)[8]) {
    const int col = k * 2048 + 8 * tid;
    if (n.fp32) {
        const float4 *p = reinterpret_cast<const float4 *>(row) + col / 4;
        const float4 a = p[0], b = p[1];
        g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
        g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
    } else {
        unpack8(*reinterpret_cast<const uint4 *>(row + 2 * col), g);
    }
    if (n.center != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            g[i] = __fadd_rn(g[i], n.center);
    }
}

// norm_scale with the weight row (when the weight scales the input) staged.
template <int R>
__device__ __forceinline__ void staged_scale(const uint4 (&q)[R][kFrags], const NormDesc &n,
                                             const uint8_t *grow, float (&sums)[2][R][kThreads / 32],
                                             int &buf, int tid, int warp, int lane, float (&r)[R]) {
    const bool in_scale = n.w != nullptr && n.input_scale;
    float p[R];
#pragma unroll
    for (int j = 0; j < R; ++j)
        p[j] = 0.0f;
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        float g[8];
        if (in_scale)
            smem_gains(n, grow, k, tid, g);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            float f[8];
            unpack8(q[j][k], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (in_scale)
                    f[i] = __fmul_rn(g[i], f[i]);
                p[j] = __fadd_rn(p[j], __fmul_rn(f[i], f[i]));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
        p[j] = warp_butterfly_sum(p[j]);
        if (lane == 0)
            sums[buf][j][warp] = p[j];
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < R; ++j) {
        float s = sums[buf][j][0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w)
            s = __fadd_rn(s, sums[buf][j][w]);
        r[j] = inv_rms(s, 0x1p-13f, n.eps);
    }
    buf ^= 1;
}

// norm_output with the weight row staged.
template <int R>
__device__ __forceinline__ void staged_output(const uint4 (&q)[R][kFrags], const NormDesc &n,
                                              const uint8_t *grow, int k, int tid, const float (&r)[R],
                                              uint4 (&o)[R]) {
    const bool weighted = n.w != nullptr;
    float g[8];
    if (weighted)
        smem_gains(n, grow, k, tid, g);
#pragma unroll
    for (int j = 0; j < R; ++j) {
        float f[8];
        unpack8(q[j][k], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (weighted && n.input_scale)
                f[i] = __fmul_rn(g[i], f[i]);
            f[i] = __fmul_rn(f[i], r[j]);
            if (weighted && !n.input_scale)
                f[i] = __fmul_rn(f[i], g[i]);
        }
        o[j] = pack8(f);
    }
}

// Buffer 0 holds the hidden weight, then layers 1, 3, ...; buffer 1 layers
// 0, 2, ...  Copy groups: [hidden], [layer 0], then one per later layer,
// issued at the top of the previous layer once every thread is past the
// buffer's last reader (the barrier after the wait).
template <int R>
__global__ void __launch_bounds__(kThreads, 2)
k1_context_norms_exs(const uint16_t *__restrict__ x, int64_t T, const NormDesc hidden,
                     const NormDesc pre, int32_t L, uint16_t *__restrict__ out, int early)
{
    extern __shared__ __align__(16) uint8_t gstage[];   // [2][kGainBytes]
    __shared__ float sums[2][R][kThreads / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row0 = (int64_t)blockIdx.x * R;
    int buf = 0;
    pdl_trigger();
    if (!early)
        pdl_wait();
    stage_gains(hidden, 0, gstage, tid);
    stage_gains(pre, 0, gstage + kGainBytes, tid);

    uint4 q[R][kFrags];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const bool live = row0 + j < T;             // missing last rows read as zeros
        const uint4 *xr = reinterpret_cast<const uint4 *>(x) + (row0 + j) * (kHidden / 8);
#pragma unroll
        for (int k = 0; k < kFrags; ++k)
            q[j][k] = live ? __ldcs(xr + k * kFragStride + tid) : make_uint4(0, 0, 0, 0);
    }
    staged_wait<1>();                               // the hidden weight (this thread's part)
    __syncthreads();
    // a1: the hidden norm, rounded to bf16 (z kept packed, in place of x)
    float r[R];
    staged_scale<R>(q, hidden, gstage, sums, buf, tid, warp, lane, r);
#pragma unroll
    for (int k = 0; k < kFrags; ++k) {
        uint4 o[R];
        staged_output<R>(q, hidden, gstage, k, tid, r, o);
#pragma unroll
        for (int j = 0; j < R; ++j)
            q[j][k] = o[j];
    }
    // a2: one inverse RMS for every layer unless the layer weight scales the input
    const bool per_layer = pre.w != nullptr && pre.input_scale;
    float r2[R];
    if (!per_layer) {
        NormDesc plain = pre;
        plain.w = nullptr;                          // the sum is of z itself
        staged_scale<R>(q, plain, nullptr, sums, buf, tid, warp, lane, r2);
    }
    for (int32_t l = 0; l < L; ++l) {
        staged_wait<0>();                           // layer l's row (this thread's part)
        __syncthreads();                            // ... everyone's; the other buffer is free
        if (l + 1 < L)
            stage_gains(pre, l + 1, gstage + ((l + 2) & 1) * kGainBytes, tid);
        const uint8_t *grow = gstage + ((l + 1) & 1) * kGainBytes;
        float rl[R];
        if (per_layer) {
            staged_scale<R>(q, pre, grow, sums, buf, tid, warp, lane, rl);
        } else {
#pragma unroll
            for (int j = 0; j < R; ++j)
                rl[j] = r2[j];
        }
#pragma unroll
        for (int k = 0; k < kFrags; ++k) {
            uint4 o[R];
            staged_output<R>(q, pre, grow, k, tid, rl, o);
#pragma unroll
            for (int j = 0; j < R; ++j)
                if (row0 + j < T)
                    reinterpret_cast<uint4 *>(out)[((int64_t)l * T + row0 + j) * (kHidden / 8) +
                                                   k * kFragStride + tid] = o[j];
        }
    }
    staged_wait<0>();                               // no copy outlives the CTA
    early_join(early);
}

template <int R>
cudaError_t launch_exs(const uint16_t *x, int64_t T, const NormDesc &hidden, const NormDesc &pre,
                       int32_t L, uint16_t *out, cudaStream_t stream, int early) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(k1_context_norms_exs<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 2 * kGainBytes);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            configured[dev] = true;
    }
    return launch_pdl(k1_context_norms_exs<R>, dim3((unsigned)((T + R - 1) / R)), dim3(kThreads),
                      (size_t)(2 * kGainBytes), stream, 1, x, T, hidden, pre, L, out, early);
}

}  // namespace

cudaError_t launch_context_norms_ex(const uint16_t *x, int64_t T, const NormDesc &hidden,
                                    const NormDesc &pre, int32_t L, uint16_t *out,
                                    cudaStream_t stream, bool early)
{
    const int ea = early ? 1 : 0;
    if (T >= kExTwoRowsFrom)                     // two rows per CTA, weights staged
        return launch_exs<2>(x, T, hidden, pre, L, out, stream, ea);
    return launch_pdl(k1_context_norms_ex<1>, dim3((unsigned)T), dim3(kThreads), 0, stream, 1, x, T,
                      hidden, pre, L, out, ea);
}

cudaError_t launch_context_norms(const uint16_t *x, int64_t T, const uint16_t *hidden_w,
                                 const uint16_t *pre_w, int32_t L, float hidden_eps, float pre_eps,
                                 uint16_t *out, cudaStream_t stream, bool early)
{
    const int ea = early ? 1 : 0;
    const dim3 block(kThreads);
    if (T >= kTwoRowsFrom) {                       // two rows per CTA
        const dim3 grid2((unsigned)((T + 1) / 2));
        if (hidden_w && pre_w)
            return launch_pdl(k1_context_norms2<true, true>, grid2, block, 0, stream, 1, x, T,
                              hidden_w, pre_w, L, hidden_eps, pre_eps, out, ea);
        if (hidden_w)
            return launch_pdl(k1_context_norms2<true, false>, grid2, block, 0, stream, 1, x, T,
                              hidden_w, pre_w, L, hidden_eps, pre_eps, out, ea);
        if (pre_w)
            return launch_pdl(k1_context_norms2<false, true>, grid2, block, 0, stream, 1, x, T,
                              hidden_w, pre_w, L, hidden_eps, pre_eps, out, ea);
        return launch_pdl(k1_context_norms2<false, false>, grid2, block, 0, stream, 1, x, T,
                          hidden_w, pre_w, L, hidden_eps, pre_eps, out, ea);
    }
    const dim3 grid((unsigned)T);
    if (hidden_w && pre_w)
        return launch_pdl(k1_context_norms<true, true>, grid, block, 0, stream, 1, x, T, hidden_w,
                          pre_w, L, hidden_eps, pre_eps, out, ea);
    if (hidden_w)
        return launch_pdl(k1_context_norms<true, false>, grid, block, 0, stream, 1, x, T, hidden_w,
                          pre_w, L, hidden_eps, pre_eps, out, ea);
    if (pre_w)
        return launch_pdl(k1_context_norms<false, true>, grid, block, 0, stream, 1, x, T, hidden_w,
                          pre_w, L, hidden_eps, pre_eps, out, ea);
    return launch_pdl(k1_context_norms<false, false>, grid, block, 0, stream, 1, x, T, hidden_w,
                      pre_w, L, hidden_eps, pre_eps, out, ea);
}

cudaError_t launch_row_prep(const uint16_t *x, int64_t T, const uint16_t *hidden_w, float eps,
                            uint16_t *z, float *r2, cudaStream_t stream)
{
    const dim3 grid((unsigned)T), block(kThreads);
    if (hidden_w)
        return launch_pdl(k1_row_prep<true>, grid, block, 0, stream, 1, x, hidden_w, eps, z, r2);
    return launch_pdl(k1_row_prep<false>, grid, block, 0, stream, 1, x, hidden_w, eps, z, r2);
}

}  // namespace rc
