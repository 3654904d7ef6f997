// common.cuh -- pieces shared by the kernels of libattn.so: the device error
// word protocol, bounded mbarrier waits, BF16 helpers and the internal
// launcher declarations.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace attn {

// Mask bits (same values as ATTN_MASK_* in include/attn.h).
constexpr int kMaskCausal = 1;
constexpr int kMaskWindow = 2;
constexpr int kMaskPadding = 4;

// Device error word: 0 = no error. A bounded wait that gives up stores
// (site << 8) | 1 with atomicCAS, so the first site that timed out is kept.
enum WaitSite : uint32_t {
    kSiteQFull = 1, kSiteKFull, kSiteVFull, kSiteKEmpty, kSiteVEmpty,
    kSiteSFull, kSitePFull, kSiteODone, kSiteDrain, kSiteSelftest
};

// Default limit of one wait, in SM clock cycles (about a second at the
// clocks these parts run at). Legitimate waits inside one CTA are
// microseconds long.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Wait until the phase of `bar` with parity `parity` completes. Gives up
// (returns false) when `*abort_flag` is set by another role of the CTA, or
// after `limit` cycles, in which case it records the site in the error word
// and raises the CTA's abort flag so that the other roles stop too.
// `abort_flag` may be NULL (the drain waits, which run after the roles have
// stopped): then only the limit ends the wait. kCluster: acquire at cluster
// scope (barriers that the other CTA of a pair signals).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned int* err,
                                             uint32_t site, long long limit = kWaitLimitCycles) {
    auto test = [&]() {
        return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const long long t0 = clock64();
    while (true) {
        if (test()) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (clock64() - t0 > limit) {
            if (abort_flag != nullptr) *abort_flag = 1;
            atomicCAS(err, 0u, (site << 8) | 1u);
            return false;
        }
    }
}

// Software 2^x for two values at once on the FMA pipe (the forward kernel
// computes part of its exponentials this way so that they do not all queue
// on the MUFU unit; the partial software exponential is the FlashAttention-4
// device P1 mentions under "What did FlashAttention-2 and -3 change?").
// Method: Cody-Waite range reduction for base 2 -- n = round(x) by adding
// 1.5 * 2^23 (the sum's low mantissa bits hold n), f = x - n in [-1/2, 1/2]
// -- then 2^f by the degree-3 polynomial 1 + c1 f + c2 f^2 + c3 f^3 whose
// coefficients minimise the maximum relative error on [-1/2, 1/2] (fitted
// by linear programming; relative error 1.02e-4, see exp2_poly_fit.py), and
// 2^n applied by adding n to the exponent field. Inputs are clamped to
// >= -127, and a result whose exponent field would fall below zero is
// returned as +0: x <= -127 (and -inf) gives +0, -127 < x < -126 a denormal
// below 2^-126.
constexpr float kExp2C1 = 0.6932829022407532f;
constexpr float kExp2C2 = 0.24221095442771912f;
constexpr float kExp2C3 = 0.055008936673402786f;

__device__ __forceinline__ float2 soft_exp2x2(float2 x) {
    constexpr float kRound = 12582912.0f;                       // 1.5 * 2^23
    x.x = fmaxf(x.x, -127.f);
    x.y = fmaxf(x.y, -127.f);
    const float2 t = __fadd2_rn(x, make_float2(kRound, kRound));
    const float2 n = __fadd2_rn(t, make_float2(-kRound, -kRound));
    const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), x);  // x - n, exact
    float2 p = __ffma2_rn(make_float2(kExp2C3, kExp2C3), f, make_float2(kExp2C2, kExp2C2));
    p = __ffma2_rn(p, f, make_float2(kExp2C1, kExp2C1));
    p = __ffma2_rn(p, f, make_float2(1.f, 1.f));
    // exponent field += n (mod 2^32: the low 9 bits of t's pattern, shifted
    // to bit 23, are n's two's complement there); a negative result -> +0.
    const uint32_t e0 = __float_as_uint(p.x) + (__float_as_uint(t.x) << 23);
    const uint32_t e1 = __float_as_uint(p.y) + (__float_as_uint(t.y) << 23);
    return make_float2(__int_as_float(max(static_cast<int>(e0), 0)),
                       __int_as_float(max(static_cast<int>(e1), 0)));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
// Exact widening of BF16 to FP32 (the BF16 bits are the high half).
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Arguments common to the forward launchers.
struct FwdArgs {
    const void* q; const void* k; const void* v;
    void* o; float* lse;
    int B, H, Nq, Nk, d;
    float scale;
    int mask_kind, window;
    const int* seqlens_k;
    unsigned int* err;     // device error word
};

// Internal launchers (return a cudaError_t from the launch; argument checks
// happen in attn_api.cu before these are called).
cudaError_t launch_fwd_f32(const FwdArgs& a, cudaStream_t stream);

struct DecodeArgs {
    const void* q; const void* k; const void* v;
    void* o; float* lse;
    int B, H, Nk, d;
    float scale;
    const int* seqlens_k;
    int num_splits;
    float* ws_o;       // [B,H,num_splits,d]
    float* ws_lse;     // [B,H,num_splits]
    unsigned int* err;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// Device address and size of decode.cu's fixed scratch array on the current
// device (looked up on first use per device).
cudaError_t decode_static_scratch(void** ptr, size_t* bytes);
struct BwdArgs {
    const void* q; const void* k; const void* v; const void* o; const void* dout;
    const float* lse;
    void* dq; void* dk; void* dv;
    int B, H, Nq, Nk, d;
    float scale;
    int mask_kind, window;
    const int* seqlens_k;
    float* ws_lse2;    // [B*H][Nq rounded up to 128]
    float* ws_dd;      // same shape
    float* ws_dq;      // [B*H][Nq rounded up to 128][d] FP32 dQ accumulator, or NULL when
                       // dQ has its own kernel (see bwd_fused_dq)
    unsigned int* err;
};
// True when attn_bwd accumulates dQ inside the keys-outer kernel for head
// dimension d (and so needs the FP32 dQ workspace).
bool bwd_fused_dq(int d);
// tdk, tdv: maps of dk and dv with the layout of tk and tv (the dK/dV
// epilogue's stores)
cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const CUtensorMap& tk64, const CUtensorMap& tv64,
                       cudaStream_t stream);
cudaError_t launch_softmax_rows(const void* x, void* y, float* lse, long long rows, int n,
                                bool bf16, cudaStream_t stream);
cudaError_t launch_fill_empty(void* o, float* lse, long long rows, int d, bool bf16,
                              cudaStream_t stream);

}  // namespace attn
