// fwd_f32.cu -- FP32 fused attention forward on the CUDA cores.
//
// The query-tile online softmax of P2 ("Implement online softmax for a whole
// tile of queries ...", "A strong answer"): every query row keeps its running
// max m, normalizer l and unnormalised accumulator a in registers while the
// CTA streams 32-key blocks of K and V through shared memory; per block
//   m' = max(m, rowmax S), m_ref = (m' == -inf ? 0 : m'),
//   alpha = exp(m - m_ref), P = exp(S - m_ref),
//   l = alpha l + P 1, a = alpha a + P V,
// and o = a / l once at the end (the single diag(l)^-1). The m_ref guard is
// the one P2 describes for rows that have not seen a key yet.
//
// Layout: D/32 threads share one query row; each owns 32 consecutive head
// dimensions of q and a. All arithmetic is FP32 with the accurate expf/logf.
#include "common.cuh"

namespace attn {
namespace {

constexpr int kThreads = 128;
constexpr int kBK = 32;   // keys per block

template <int D>
__global__ void __launch_bounds__(kThreads)
fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
               const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
               int H, int Nq, int Nk, float scale, int mask_kind, int window,
               const int* __restrict__ seqlens_k) {
    constexpr int TPR = D / 32;               // threads per query row
    constexpr int RB = kThreads / TPR;        // query rows per CTA
    __shared__ __align__(16) float Ks[kBK][D];
    __shared__ __align__(16) float Vs[kBK][D];

    const int b = blockIdx.z, h = blockIdx.y;
    const long long bh = static_cast<long long>(b) * H + h;
    const int row0 = blockIdx.x * RB;
    const int sub = threadIdx.x % TPR;
    const int i = row0 + threadIdx.x / TPR;   // this thread's query row

    int Lk = Nk;
    if (mask_kind & kMaskPadding) Lk = min(max(seqlens_k[b], 0), Nk);
    const bool causal = (mask_kind & (kMaskCausal | kMaskWindow)) != 0;
    const bool windowed = (mask_kind & kMaskWindow) != 0;

    // Key range that any row of this CTA can see (blocks outside are skipped).
    const int row_last = min(row0 + RB, Nq) - 1;
    int key_hi = Lk;
    if (causal) key_hi = min(key_hi, row_last + 1);
    int key_lo = windowed ? max(0, row0 - window + 1) : 0;
    key_lo = (key_lo / kBK) * kBK;

    float qr[32], acc[32];
    const float* qrow = q + (bh * Nq + min(i, Nq - 1)) * D + sub * 32;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        qr[e] = (i < Nq) ? qrow[e] : 0.f;
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    const float* kh = k + bh * static_cast<long long>(Nk) * D;
    const float* vh = v + bh * static_cast<long long>(Nk) * D;
    for (int kb = key_lo; kb < key_hi; kb += kBK) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kBK * D / 4; idx += kThreads) {
            const int kk = idx / (D / 4), c = idx % (D / 4);
            const int key = kb + kk;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (key < Nk) {
                kv = reinterpret_cast<const float4*>(kh + static_cast<long long>(key) * D)[c];
                vv = reinterpret_cast<const float4*>(vh + static_cast<long long>(key) * D)[c];
            }
            reinterpret_cast<float4*>(&Ks[kk][0])[c] = kv;
            reinterpret_cast<float4*>(&Vs[kk][0])[c] = vv;
        }
        __syncthreads();

        float s[kBK];
        float bmax = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) part = fmaf(qr[e], Ks[kk][sub * 32 + e], part);
#pragma unroll
            for (int off = 1; off < TPR; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            const int key = kb + kk;
            bool vis = key < Lk;
            if (causal) vis = vis && key <= i;
            if (windowed) vis = vis && key > i - window;
            s[kk] = vis ? part * scale : -INFINITY;
            bmax = fmaxf(bmax, s[kk]);
        }
        const float m_new = fmaxf(m, bmax);
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = expf(m - m_ref);
        float psum = 0.f;
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            s[kk] = expf(s[kk] - m_ref);
            psum += s[kk];
        }
        l = alpha * l + psum;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            float a = alpha * acc[e];
#pragma unroll
            for (int kk = 0; kk < kBK; ++kk) a = fmaf(s[kk], Vs[kk][sub * 32 + e], a);
            acc[e] = a;
        }
        m = m_new;
    }

    if (i < Nq) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        float* orow = o + (bh * Nq + i) * D + sub * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(orow + e) =
                make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv);
        if (lse != nullptr && sub == 0)
            lse[bh * Nq + i] = (l > 0.f) ? m + logf(l) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs& a, cudaStream_t stream) {
    const int rb = kThreads / (a.d / 32);
    dim3 grid((a.Nq + rb - 1) / rb, a.H, a.B);
    if (a.d == 64) {
        fwd_f32_kernel<64><<<grid, kThreads, 0, stream>>>(
            static_cast<const float*>(a.q), static_cast<const float*>(a.k),
            static_cast<const float*>(a.v), static_cast<float*>(a.o), a.lse, a.H, a.Nq, a.Nk,
            a.scale, a.mask_kind, a.window, a.seqlens_k);
    } else {
        fwd_f32_kernel<128><<<grid, kThreads, 0, stream>>>(
            static_cast<const float*>(a.q), static_cast<const float*>(a.k),
            static_cast<const float*>(a.v), static_cast<float*>(a.o), a.lse, a.H, a.Nq, a.Nk,
            a.scale, a.mask_kind, a.window, a.seqlens_k);
    }
    return cudaGetLastError();
}

}  // namespace attn
