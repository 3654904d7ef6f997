// decode.cu -- split-KV decode (Flash-Decoding): one query row per (b, h),
// the key range cut into contiguous chunks that run on separate CTAs, then a
// reduction that merges the chunks.
//
// Launch 1, decode_split_kernel: grid (num_splits, H, B). Each CTA runs the
// single-query online recurrence of P1 ("Derive online softmax, prove it is
// exact, ...", "A strong answer") over its chunk -- running max m, normalizer
// l and unnormalised output a, rescaled by exp(m_old - m_new) whenever a
// batch of keys raises the max -- and writes the chunk's normalised output
// o_s = a / l and log-sum-exp lse_s = m + log l (the per-chunk form that P3
// "Online softmax", "Trade-offs and edge cases", attributes to Flash-
// Decoding). An empty chunk writes o_s = 0, lse_s = -inf.
//
// Launch 2, decode_combine_kernel: grid (H, B). Merges the chunks of one
// (b, h) with the associative rule of P3 "Step 4": m* = max_s lse_s,
// w_s = exp(lse_s - m*), o = sum w_s o_s / sum w_s, lse = m* + log sum w_s.
// It is a programmatic dependent launch: its CTAs may be scheduled while
// the split kernel's last wave runs, and wait (griddepcontrol.wait) for
// that grid's completion and memory before reading any partial, which
// hides most of the gap between the two launches.
//
// The work is one multiply-add per key element for the scores and one for
// the output: the split kernel is bound by HBM bandwidth. Each warp streams
// its keys with 16-byte non-allocating loads, 16 keys (d = 128) per batch,
// so every lane has 16 independent loads in flight per batch.
#include <mutex>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kSplitThreads = 256;
constexpr int kWarps = kSplitThreads / 32;
constexpr int kUnroll = 8;                   // load instructions per batch per tensor
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ float dot8(const float* qf, uint4 kw) {
    float s = qf[0] * bf16lo_to_f32(kw.x);
    s = fmaf(qf[1], bf16hi_to_f32(kw.x), s);
    s = fmaf(qf[2], bf16lo_to_f32(kw.y), s);
    s = fmaf(qf[3], bf16hi_to_f32(kw.y), s);
    s = fmaf(qf[4], bf16lo_to_f32(kw.z), s);
    s = fmaf(qf[5], bf16hi_to_f32(kw.z), s);
    s = fmaf(qf[6], bf16lo_to_f32(kw.w), s);
    s = fmaf(qf[7], bf16hi_to_f32(kw.w), s);
    return s;
}

__device__ __forceinline__ void axpy8(float* acc, float p, uint4 vw) {
    acc[0] = fmaf(p, bf16lo_to_f32(vw.x), acc[0]);
    acc[1] = fmaf(p, bf16hi_to_f32(vw.x), acc[1]);
    acc[2] = fmaf(p, bf16lo_to_f32(vw.y), acc[2]);
    acc[3] = fmaf(p, bf16hi_to_f32(vw.y), acc[3]);
    acc[4] = fmaf(p, bf16lo_to_f32(vw.z), acc[4]);
    acc[5] = fmaf(p, bf16hi_to_f32(vw.z), acc[5]);
    acc[6] = fmaf(p, bf16lo_to_f32(vw.w), acc[6]);
    acc[7] = fmaf(p, bf16hi_to_f32(vw.w), acc[7]);
}

// Scores are kept in the log2 domain: s2 = (scale * log2 e) * <q, k>, so
// exp(s - m) = exp2(s2 - m2).
template <int D>
__global__ void __launch_bounds__(kSplitThreads)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, float* __restrict__ ws_o,
                    float* __restrict__ ws_lse, int H, int Nk, int split_len, int num_splits,
                    float scale_log2, const int* __restrict__ seqlens_k) {
    constexpr int LPK = D / 8;        // lanes per key row (16 bytes each)
    constexpr int KPI = 32 / LPK;     // keys per warp load instruction
    constexpr int KPB = KPI * kUnroll;  // keys per batch per warp
    // the combine launch may start now; it waits for this grid to complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    __shared__ float sm_m[kWarps], sm_l[kWarps];
    __shared__ __align__(16) float sm_acc[kWarps][D];

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const long long bh = static_cast<long long>(b) * H + h;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane % LPK, slot = lane / LPK;

    int Lk = Nk;
    if (seqlens_k != nullptr) Lk = min(max(seqlens_k[b], 0), Nk);
    const int c_begin = split * split_len;
    const int c_end = min(c_begin + split_len, Lk);
    const int c_len = max(c_end - c_begin, 0);
    // contiguous sub-range per warp, in whole batches
    const int per_warp = ((c_len + kWarps * KPB - 1) / (kWarps * KPB)) * KPB;
    const int w_begin = c_begin + warp * per_warp;
    const int w_end = min(w_begin + per_warp, c_end);

    float qf[8];
    {
        const uint4 qw = *reinterpret_cast<const uint4*>(q + bh * D + sub * 8);
        qf[0] = bf16lo_to_f32(qw.x) * scale_log2; qf[1] = bf16hi_to_f32(qw.x) * scale_log2;
        qf[2] = bf16lo_to_f32(qw.y) * scale_log2; qf[3] = bf16hi_to_f32(qw.y) * scale_log2;
        qf[4] = bf16lo_to_f32(qw.z) * scale_log2; qf[5] = bf16hi_to_f32(qw.z) * scale_log2;
        qf[6] = bf16lo_to_f32(qw.w) * scale_log2; qf[7] = bf16hi_to_f32(qw.w) * scale_log2;
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float m = -INFINITY, l = 0.f;

    const __nv_bfloat16* kh = k + bh * static_cast<long long>(Nk) * D + sub * 8;
    const __nv_bfloat16* vh = v + bh * static_cast<long long>(Nk) * D + sub * 8;
    for (int base = w_begin; base < w_end; base += KPB) {
        uint4 kw[kUnroll], vw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + u * KPI + slot;
            if (key < w_end) {
                kw[u] = ldg_stream(kh + static_cast<long long>(key) * D);
                vw[u] = ldg_stream(vh + static_cast<long long>(key) * D);
            } else {
                kw[u] = make_uint4(0, 0, 0, 0);
                vw[u] = kw[u];
            }
        }
        float s[kUnroll];
        float bmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float part = dot8(qf, kw[u]);
#pragma unroll
            for (int off = LPK / 2; off >= 1; off >>= 1)
                part += __shfl_xor_sync(0xffffffffu, part, off);
            const int key = base + u * KPI + slot;
            s[u] = (key < w_end) ? part : -INFINITY;
            bmax = fmaxf(bmax, s[u]);
        }
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1)
            bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
        const float m_new = fmaxf(m, bmax);
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ptx::ex2(m - m_ref);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float p = ptx::ex2(s[u] - m_ref);
            l += p;
            axpy8(acc, p, vw[u]);
        }
        m = m_new;
    }
    // Sum the key slots of the warp (they share m): lanes with equal `sub`.
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
        l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    }
    if (lane == 0) { sm_m[warp] = m; sm_l[warp] = l; }
    if (slot == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) sm_acc[warp][sub * 8 + e] = acc[e];
    }
    __syncthreads();
    // Merge the warps' (m, l, a) with the same rescaling rule.
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
    const float M_ref = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) L += sm_l[w] * ptx::ex2(sm_m[w] - M_ref);
    const long long slot_idx = bh * num_splits + split;
    for (int e = threadIdx.x; e < D; e += kSplitThreads) {
        float A = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) A += sm_acc[w][e] * ptx::ex2(sm_m[w] - M_ref);
        ws_o[slot_idx * D + e] = (L > 0.f) ? A / L : 0.f;
    }
    if (threadIdx.x == 0)
        ws_lse[slot_idx] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

// 128 threads per (b, h). The partial outputs, the bulk of what the merge
// reads, arrive as 16-byte vectors: D / 4 lanes cover one split's row of D
// FP32 values, and the 128 threads take 128 / (D / 4) split rows at a time,
// so every warp load is one fully used 512-byte (D = 128) or two 256-byte
// (D = 64) contiguous segments. The rows' sums meet in shared memory.
constexpr int kCombineThreads = 128;

template <int D>
__global__ void __launch_bounds__(kCombineThreads)
decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int H,
                      int num_splits) {
    constexpr int LPR = D / 4;                       // lanes per split row (one float4 each)
    constexpr int RPI = kCombineThreads / LPR;       // split rows per iteration
    extern __shared__ float sm_w[];                  // num_splits weights
    __shared__ __align__(16) float4 part[RPI][LPR];
    __shared__ float red[kCombineThreads / 32];
    __shared__ float bcast;
    // every partial is written by the split grid, which must have completed
    // (a no-op when launched without the programmatic attribute)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long bh = static_cast<long long>(blockIdx.y) * H + blockIdx.x;
    const float* lp = ws_lse + bh * num_splits;
    const int tid = threadIdx.x;
    // m* = max_s lse_s
    float mx = -INFINITY;
    for (int s = tid; s < num_splits; s += kCombineThreads) mx = fmaxf(mx, lp[s]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (tid % 32 == 0) red[tid / 32] = mx;
    __syncthreads();
    if (tid == 0) {
        float t = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCombineThreads / 32; ++w) t = fmaxf(t, red[w]);
        bcast = t;
    }
    __syncthreads();
    const float M = bcast;
    const float M_ref = (M == -INFINITY) ? 0.f : M;
    // w_s = exp(lse_s - m*)
    for (int s = tid; s < num_splits; s += kCombineThreads)
        sm_w[s] = ptx::ex2((lp[s] - M_ref) * kLog2e);
    __syncthreads();
    // sum_s w_s o_s, 16 bytes per lane per split row
    const int r = tid / LPR, c = tid % LPR;
    const float4* op = reinterpret_cast<const float4*>(ws_o + bh * num_splits * D) + c;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    for (int s = r; s < num_splits; s += RPI) {
        const float w = sm_w[s];
        const float4 x = op[static_cast<long long>(s) * LPR];
        a.x = fmaf(w, x.x, a.x);
        a.y = fmaf(w, x.y, a.y);
        a.z = fmaf(w, x.z, a.z);
        a.w = fmaf(w, x.w, a.w);
    }
    part[r][c] = a;
    if (tid < 32) {
        for (int s = tid; s < num_splits; s += 32) W += sm_w[s];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
        if (tid == 0) bcast = W;
    }
    __syncthreads();
    if (tid < LPR) {
        float4 t = part[0][tid];
#pragma unroll
        for (int rr = 1; rr < RPI; ++rr) {
            const float4 u = part[rr][tid];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const float Wt = bcast;
        const float inv = Wt > 0.f ? 1.f / Wt : 0.f;
        uint2 packed;
        packed.x = pack_bf16x2(t.x * inv, t.y * inv);
        packed.y = pack_bf16x2(t.z * inv, t.w * inv);
        *reinterpret_cast<uint2*>(o + bh * D + 4 * tid) = packed;
        if (lse != nullptr && tid == 0) lse[bh] = (Wt > 0.f) ? M + logf(Wt) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    const int split_len = (a.Nk + a.num_splits - 1) / a.num_splits;
    const float scale_log2 = a.scale * kLog2e;
    dim3 g1(a.num_splits, a.H, a.B), g2(a.H, a.B);
    const size_t smem2 = sizeof(float) * a.num_splits;
    const auto* q = static_cast<const __nv_bfloat16*>(a.q);
    const auto* k = static_cast<const __nv_bfloat16*>(a.k);
    const auto* v = static_cast<const __nv_bfloat16*>(a.v);
    auto* o = static_cast<__nv_bfloat16*>(a.o);
    // the combine as a programmatic dependent launch of the split grid
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = g2;
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = smem2;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* ws_o = a.ws_o;
    const float* ws_lse = a.ws_lse;
    float* lse = a.lse;
    const int H = a.H, ns = a.num_splits;
    if (a.d == 64) {
        decode_split_kernel<64><<<g1, kSplitThreads, 0, stream>>>(
            q, k, v, a.ws_o, a.ws_lse, a.H, a.Nk, split_len, a.num_splits, scale_log2, a.seqlens_k);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, ws_o, ws_lse, o, lse, H, ns);
    }
    decode_split_kernel<128><<<g1, kSplitThreads, 0, stream>>>(
        q, k, v, a.ws_o, a.ws_lse, a.H, a.Nk, split_len, a.num_splits, scale_log2, a.seqlens_k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, ws_o, ws_lse, o, lse, H, ns);
}

// ---------------------------------------------------------------------------
// Decode without caller-provided scratch.
//
// Some callers cannot hand this library a device buffer for the split
// partials: a serving process that has reserved all device memory for its own
// pool and forbids allocation on the request path, or a caller that must not
// call cudaMalloc/cudaFree there because those calls can synchronise the
// device and stall work on other streams. For them the split partials live in
// the fixed array below instead of a workspace argument.
//
// Limits and sharing:
//   * kStaticScratchBytes (4 MiB) is the whole array; it holds the partials
//     of B * H * num_splits (b, h, split) slots: d FP32 outputs per slot plus
//     one FP32 log-sum-exp per slot, laid out exactly like the workspace of
//     attn_decode_splitkv (attn_decode_workspace_bytes). Problems that need
//     more are rejected.
//   * Every GPU that loads libattn.so holds this array until the process exits.
//   * All calls on a device share the one array and it keeps the last call's
//     contents. Nothing in it has to start at zero: the split launch writes
//     every slot the combine launch then reads. Two calls whose kernels
//     overlap on the GPU (for example on two streams without ordering between
//     them) race on the array and give wrong results.
//   * In host code the name g_decode_scratch is only a host-side stand-in for
//     the device array; its device address is looked up once per device with
//     cudaGetSymbolAddress (below), with that device current.
// ---------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

cudaError_t decode_static_scratch(void** ptr, size_t* bytes) {
    static std::mutex mu;
    static void* cache[128] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        cache[dev] = p;
    }
    *ptr = cache[dev];
    *bytes = kStaticScratchBytes;
    return cudaSuccess;
}

}  // namespace attn
