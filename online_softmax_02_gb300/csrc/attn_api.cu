// attn_api.cu -- the C interface of libattn.so (declared in include/attn.h):
// argument checks, TMA tensor-map encoding, launch, the per-device error
// word, and the small utility kernels (empty-row fill, bounded-wait
// self-test).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "common.cuh"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace attn {

cudaError_t launch_fwd_sm103_maps(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& to, bool pair,
                                  cudaStream_t stream);
cudaError_t launch_fwd_fp8_maps(const FwdArgs& a, float descale_q, float descale_k,
                                float descale_v, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t stream);

namespace {

// 1: the BF16 forward at d = 128 runs on CTA pairs (cta_group::2: each K/V
// block is split between two SMs and every MMA spans both). 0 (default): the
// one-CTA kernel, which d = 64 and the E4M3 forward always use. The pair form
// measured slower on GB300 (prefill B1 H64 8192^2: 1.65 against 1.34 ms;
// causal 0.92 against 0.70): the forward's pace is set by the softmax -> P
// -> MMA hand-off, and in a pair each hand-off crosses to the other SM and
// waits for the slower of two softmaxes.
#ifndef ATTN_FWD_PAIR
#define ATTN_FWD_PAIR 0
#endif
constexpr bool kFwdPair = ATTN_FWD_PAIR != 0;

__device__ unsigned int g_err_word = 0;   // see WaitSite in common.cuh

thread_local std::string t_last_error;

attn_status_t fail(attn_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

attn_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device address of the error word on the current device (cached per device).
attn_status_t err_word(unsigned int** out) {
    static std::mutex mu;
    static unsigned int* cache[128] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 128) return fail(ATTN_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_err_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        cache[dev] = static_cast<unsigned int*>(p);
    }
    *out = cache[dev];
    return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D tensor map over [B*H][rows][d] with 128-byte swizzle and a box of one
// swizzle atom row (128 bytes: 64 BF16 or 128 8-bit head dims) x box_rows x 1.
attn_status_t encode_3d(CUtensorMap* m, const void* ptr, int d, int rows, long long bh,
                        bool one_byte, unsigned box_rows = 128) {
    auto fn = encode_fn();
    if (fn == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
    const cuuint64_t esz = one_byte ? 1 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(bh)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esz,
                             static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(d) * esz};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, one_byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ATTN_OK;
}

attn_status_t encode_bf16_3d(CUtensorMap* m, const void* ptr, int d, int rows, long long bh) {
    return encode_3d(m, ptr, d, rows, bh, false);
}

__global__ void fill_empty_kernel(void* o, float* lse, long long rows, int d, int is_bf16) {
    const long long n = rows * d;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        if (is_bf16) static_cast<__nv_bfloat16*>(o)[i] = __float2bfloat16_rn(0.f);
        else static_cast<float*>(o)[i] = 0.f;
        if (lse != nullptr && i % d == 0) lse[i / d] = -INFINITY;
    }
}

__global__ void exp2_soft_kernel(const float* x, float* y, long long n) {
    for (long long i = 2 * (blockIdx.x * (long long)blockDim.x + threadIdx.x); i < n;
         i += 2 * (long long)gridDim.x * blockDim.x) {
        const float2 r = soft_exp2x2(make_float2(x[i], i + 1 < n ? x[i + 1] : 0.f));
        y[i] = r.x;
        if (i + 1 < n) y[i + 1] = r.y;
    }
}

__global__ void selftest_wait_kernel(unsigned int* err, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`: the wait must give up after `limit`.
    wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, err, kSiteSelftest, limit);
}

// Checks shared by attn_fwd and attn_fwd_f32. Returns ATTN_OK and sets
// *empty when there is nothing to compute.
attn_status_t check_fwd(const void* q, const void* k, const void* v, const void* o, int B, int H,
                        int Nq, int Nk, int d, float scale, int mask_kind, int window,
                        const int* seqlens_k, bool* nothing) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d Nq=%d Nk=%d)", B, H, Nq, Nk);
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_WINDOW | ATTN_MASK_PADDING))
        return fail(ATTN_ERR_INVALID_ARG, "unknown mask bits 0x%x", mask_kind);
    if ((mask_kind & ATTN_MASK_WINDOW) && window < 1)
        return fail(ATTN_ERR_INVALID_ARG, "window must be >= 1 with ATTN_MASK_WINDOW");
    if (((mask_kind & ATTN_MASK_PADDING) != 0) != (seqlens_k != nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "seqlens_k must be given iff ATTN_MASK_PADDING is set");
    if (B > 65535 || H > 65535)
        return fail(ATTN_ERR_UNSUPPORTED, "B and H must be <= 65535");
    *nothing = (static_cast<long long>(B) * H * Nq == 0);
    if (*nothing) return ATTN_OK;
    if (q == nullptr || o == nullptr) return fail(ATTN_ERR_INVALID_ARG, "q and o must not be NULL");
    if (Nk > 0 && (k == nullptr || v == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "k and v must not be NULL");
    if (!aligned16(q) || !aligned16(o) || (Nk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    return ATTN_OK;
}

// The BF16 forward on device buffers, after the argument checks.
attn_status_t fwd_bf16_launch(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Nq, int Nk, int d, float scale, int mask_kind,
                              int window, const int* seqlens_k, cudaStream_t s) {
    attn_status_t st;
    const long long rows = static_cast<long long>(B) * H * Nq;
    if (Nk == 0) {
        cudaError_t e = launch_fill_empty(o, lse, rows, d, true, s);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "fill kernel launch");
    }
    unsigned int* err = nullptr;
    if ((st = err_word(&err)) != ATTN_OK) return st;
    CUtensorMap tq, tk, tv, to;
    const long long bh = static_cast<long long>(B) * H;
    // d = 128 runs on CTA pairs, each CTA loading 64 keys of every K block
    const bool pair = kFwdPair && d == 128;
    if ((st = encode_bf16_3d(&tq, q, d, Nq, bh)) != ATTN_OK) return st;
    if ((st = encode_3d(&tk, k, d, Nk, bh, false, pair ? 64 : 128)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&tv, v, d, Nk, bh)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&to, o, d, Nq, bh)) != ATTN_OK) return st;   // the epilogue's stores
    FwdArgs a{q, k, v, o, lse, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k, err};
    cudaError_t e = launch_fwd_sm103_maps(a, tq, tk, tv, to, pair, s);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_fwd kernel launch");
}

}  // namespace
}  // namespace attn

using namespace attn;

ATTN_API attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Nq, int Nk, int d, float scale, int mask_kind,
                                int window, const int* seqlens_k, attn_stream_t stream) {
    bool nothing = false;
    attn_status_t st = check_fwd(q, k, v, o, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k,
                                 &nothing);
    if (st != ATTN_OK || nothing) return st;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    return fwd_bf16_launch(q, k, v, o, lse, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k,
                           static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// attn_fwd_host: the forward on host-resident inputs and outputs.
//
// The (b, h) heads are cut into contiguous groups; each group is copied into
// one of `slots` device buffer sets of the caller's workspace, computed by the
// same kernel as attn_fwd, and copied back, so that the copy-in of one group,
// the kernel of another and the copy-out of a third overlap (only Q, K, V and
// O cross the host link, as only they cross HBM in the fused method).
// Streams and events are the library's own, created once per device.
// ---------------------------------------------------------------------------
namespace attn {
namespace {

constexpr int kMaxHostSlots = 8;

struct HostLayout {
    long long bh = 0, per = 0, groups = 0;
    int slots = 0;
    size_t q = 0, kv = 0, o = 0, lse = 0, slot = 0, lens = 0, total = 0;
};

bool host_layout(int B, int H, int Nq, int Nk, int d, int groups, int slots, HostLayout* L) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || (d != 64 && d != 128) || groups < 1 ||
        slots < 1 || slots > kMaxHostSlots)
        return false;
    L->bh = static_cast<long long>(B) * H;
    if (L->bh == 0) return true;
    const long long g = std::min<long long>(groups, L->bh);
    L->per = (L->bh + g - 1) / g;
    L->groups = (L->bh + L->per - 1) / L->per;
    L->slots = static_cast<int>(std::min<long long>(slots, L->groups));
    const size_t per = static_cast<size_t>(L->per);
    L->q = align256(per * Nq * d * 2);
    L->kv = align256(per * Nk * d * 2);
    L->o = L->q;
    L->lse = align256(per * Nq * sizeof(float));
    L->slot = L->q + 2 * L->kv + L->o + L->lse;
    L->lens = align256(static_cast<size_t>(L->bh) * sizeof(int) + static_cast<size_t>(B) * sizeof(int));
    L->total = L->slots * L->slot + L->lens;
    return true;
}

// The library's copy and compute streams and their events on one device.
struct HostStreams {
    std::mutex mu;                       // one enqueue at a time per device
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, run[kMaxHostSlots] = {};
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t ev_in[kMaxHostSlots] = {}, ev_run[kMaxHostSlots] = {}, ev_out[kMaxHostSlots] = {};
};

attn_status_t host_streams(HostStreams** out) {
    static std::mutex create_mu;
    static HostStreams per_device[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 128) return fail(ATTN_ERR_UNSUPPORTED, "device index %d", dev);
    HostStreams& h = per_device[dev];
    std::lock_guard<std::mutex> lock(create_mu);
    if (!h.ready) {
        auto mk_s = [](cudaStream_t* s) { return cudaStreamCreateWithFlags(s, cudaStreamNonBlocking); };
        auto mk_e = [](cudaEvent_t* ev) { return cudaEventCreateWithFlags(ev, cudaEventDisableTiming); };
        if ((e = mk_s(&h.in)) != cudaSuccess || (e = mk_s(&h.out)) != cudaSuccess ||
            (e = mk_e(&h.start)) != cudaSuccess || (e = mk_e(&h.done)) != cudaSuccess)
            return cuda_fail(e, "creating the host pipeline's streams");
        for (int i = 0; i < kMaxHostSlots; ++i)
            if ((e = mk_s(&h.run[i])) != cudaSuccess || (e = mk_e(&h.ev_in[i])) != cudaSuccess ||
                (e = mk_e(&h.ev_run[i])) != cudaSuccess || (e = mk_e(&h.ev_out[i])) != cudaSuccess)
                return cuda_fail(e, "creating the host pipeline's streams");
        h.ready = true;
    }
    *out = &h;
    return ATTN_OK;
}

// The groups' sizes in heads, in order: full groups of `per` heads, except
// that when there are at least four full groups' worth of heads (and a full
// group has 4 or more) the first two groups take a quarter and a half of a
// full group and the last two a half and a quarter. The first kernel then
// starts after a short copy and the last copy-back follows a short kernel:
// the pipeline's fill and drain, when the host link is not busy both ways,
// shrink. Prefill B1 H64 8192^2 on GB300, whose host link moves the whole
// job (403 MB in, 136 MB out) in 2.07 ms: 16 even groups 2.38 ms, 4 groups
// 2.60 ms even and 2.275 ms with this ramp; a longer ramp (an eighth first,
// or halving down to one head) measured 2.28-2.46 ms -- groups of one or
// two heads launch kernels too small to fill the GPU.
int host_group_sizes(long long bh, long long per, long long* sizes, int cap) {
    int n = 0;
    auto push = [&](long long v) {
        if (n < cap && sizes != nullptr) sizes[n] = v;
        ++n;
    };
    const bool ramp = per >= 4 && bh >= 4 * per;
    const long long quarter = (per + 3) / 4, half = (per + 1) / 2;
    long long left = bh;
    if (ramp) {
        push(quarter);
        push(half);
        left -= 2 * (quarter + half);                 // and the mirror at the end
    }
    while (left > 0) {
        const long long g = std::min(per, left);
        push(g);
        left -= g;
    }
    if (ramp) {
        push(half);
        push(quarter);
    }
    return n;
}

// lens[b * H + h] = seqlens_k[b]: one key length per head, so that any group
// of heads is a batch of one-head problems.
__global__ void expand_seqlens_kernel(const int* __restrict__ src, int* __restrict__ dst,
                                      long long bh, int H) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < bh;
         i += (long long)gridDim.x * blockDim.x)
        dst[i] = src[i / H];
}

}  // namespace
}  // namespace attn

ATTN_API size_t attn_fwd_host_workspace_bytes(int B, int H, int Nq, int Nk, int d, int groups,
                                              int slots) {
    HostLayout L;
    if (!host_layout(B, H, Nq, Nk, d, groups, slots, &L)) return 0;
    return L.total;
}

ATTN_API int attn_fwd_host_groups(int B, int H, int groups) {
    if (B < 0 || H < 0 || groups < 1) return -1;
    const long long bh = static_cast<long long>(B) * H;
    if (bh == 0) return 0;
    const long long g = std::min<long long>(groups, bh);
    return host_group_sizes(bh, (bh + g - 1) / g, nullptr, 0);
}

ATTN_API attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                                     int mask_kind, int window, const int* seqlens_k, int groups,
                                     int slots, void* workspace, size_t workspace_bytes,
                                     attn_stream_t stream) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d Nq=%d Nk=%d)", B, H, Nq, Nk);
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_WINDOW | ATTN_MASK_PADDING))
        return fail(ATTN_ERR_INVALID_ARG, "unknown mask bits 0x%x", mask_kind);
    if ((mask_kind & ATTN_MASK_WINDOW) && window < 1)
        return fail(ATTN_ERR_INVALID_ARG, "window must be >= 1 with ATTN_MASK_WINDOW");
    const bool padded = (mask_kind & ATTN_MASK_PADDING) != 0;
    if (padded != (seqlens_k != nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "seqlens_k must be given iff ATTN_MASK_PADDING is set");
    if (groups < 1) return fail(ATTN_ERR_INVALID_ARG, "groups must be >= 1");
    if (slots < 1 || slots > kMaxHostSlots)
        return fail(ATTN_ERR_INVALID_ARG, "slots must be in [1, %d]", kMaxHostSlots);
    HostLayout L;
    host_layout(B, H, Nq, Nk, d, groups, slots, &L);
    if (L.bh == 0 || Nq == 0) return ATTN_OK;
    if (L.per > 65535) return fail(ATTN_ERR_UNSUPPORTED, "more than 65535 heads per group");
    if (q == nullptr || o == nullptr || (Nk > 0 && (k == nullptr || v == nullptr)))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must not be NULL");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 1u)
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 2-byte aligned");
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (workspace == nullptr || workspace_bytes < L.total)
        return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", L.total,
                    workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");

    HostStreams* hs = nullptr;
    attn_status_t st = host_streams(&hs);
    if (st != ATTN_OK) return st;
    std::lock_guard<std::mutex> lock(hs->mu);
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    cudaError_t e;
#define ATTN_HOST_CHECK(call, what)                          \
    do {                                                     \
        if ((e = (call)) != cudaSuccess) return cuda_fail(e, what); \
    } while (0)
    // every stream of the pipeline starts after the work queued on the caller's
    ATTN_HOST_CHECK(cudaEventRecord(hs->start, caller), "cudaEventRecord");
    ATTN_HOST_CHECK(cudaStreamWaitEvent(hs->in, hs->start, 0), "cudaStreamWaitEvent");
    ATTN_HOST_CHECK(cudaStreamWaitEvent(hs->out, hs->start, 0), "cudaStreamWaitEvent");
    for (int i = 0; i < L.slots; ++i)
        ATTN_HOST_CHECK(cudaStreamWaitEvent(hs->run[i], hs->start, 0), "cudaStreamWaitEvent");

    char* ws = static_cast<char*>(workspace);
    int* lens = reinterpret_cast<int*>(ws + L.slots * L.slot);       // [B*H], then [B]
    if (padded) {
        int* lens_b = lens + L.bh;
        ATTN_HOST_CHECK(cudaMemcpyAsync(lens_b, seqlens_k, sizeof(int) * B, cudaMemcpyHostToDevice,
                                        hs->in), "copy of seqlens_k");
        const int blocks = static_cast<int>(std::min<long long>((L.bh + 255) / 256, 1024));
        expand_seqlens_kernel<<<blocks, 256, 0, hs->in>>>(lens_b, lens, L.bh, H);
        ATTN_HOST_CHECK(cudaGetLastError(), "seqlens kernel launch");
    }
    const size_t qrow = static_cast<size_t>(Nq) * d * 2, krow = static_cast<size_t>(Nk) * d * 2;
    const int ngroups = host_group_sizes(L.bh, L.per, nullptr, 0);
    std::vector<long long> sizes(static_cast<size_t>(ngroups));
    host_group_sizes(L.bh, L.per, sizes.data(), ngroups);
    long long a = 0;                                   // first head of group c
    for (int c = 0; c < ngroups; a += sizes[c], ++c) {
        const long long n = sizes[c];
        const int si = c % L.slots;
        char* sq = ws + si * L.slot;
        char* sk = sq + L.q;
        char* sv = sk + L.kv;
        char* so = sv + L.kv;
        float* sl = reinterpret_cast<float*>(so + L.o);
        if (c >= L.slots)   // the slot's previous group has been copied out
            ATTN_HOST_CHECK(cudaStreamWaitEvent(hs->in, hs->ev_out[si], 0), "cudaStreamWaitEvent");
        ATTN_HOST_CHECK(cudaMemcpyAsync(sq, static_cast<const char*>(q) + a * qrow, n * qrow,
                                        cudaMemcpyHostToDevice, hs->in), "copy of q");
        if (krow > 0) {
            ATTN_HOST_CHECK(cudaMemcpyAsync(sk, static_cast<const char*>(k) + a * krow, n * krow,
                                            cudaMemcpyHostToDevice, hs->in), "copy of k");
            ATTN_HOST_CHECK(cudaMemcpyAsync(sv, static_cast<const char*>(v) + a * krow, n * krow,
                                            cudaMemcpyHostToDevice, hs->in), "copy of v");
        }
        ATTN_HOST_CHECK(cudaEventRecord(hs->ev_in[si], hs->in), "cudaEventRecord");
        cudaStream_t run = hs->run[si];
        ATTN_HOST_CHECK(cudaStreamWaitEvent(run, hs->ev_in[si], 0), "cudaStreamWaitEvent");
        // the group as H = n heads of one batch, or, with padding, as n
        // one-head batches carrying their own key lengths
        st = fwd_bf16_launch(sq, sk, sv, so, lse != nullptr ? sl : nullptr,
                             padded ? static_cast<int>(n) : 1, padded ? 1 : static_cast<int>(n),
                             Nq, Nk, d, scale, mask_kind, window, padded ? lens + a : nullptr, run);
        if (st != ATTN_OK) return st;
        ATTN_HOST_CHECK(cudaEventRecord(hs->ev_run[si], run), "cudaEventRecord");
        ATTN_HOST_CHECK(cudaStreamWaitEvent(hs->out, hs->ev_run[si], 0), "cudaStreamWaitEvent");
        ATTN_HOST_CHECK(cudaMemcpyAsync(static_cast<char*>(o) + a * qrow, so, n * qrow,
                                        cudaMemcpyDeviceToHost, hs->out), "copy of o");
        if (lse != nullptr)
            ATTN_HOST_CHECK(cudaMemcpyAsync(lse + a * Nq, sl, n * Nq * sizeof(float),
                                            cudaMemcpyDeviceToHost, hs->out), "copy of lse");
        ATTN_HOST_CHECK(cudaEventRecord(hs->ev_out[si], hs->out), "cudaEventRecord");
    }
    // the caller's stream continues once the last copy back has landed
    ATTN_HOST_CHECK(cudaEventRecord(hs->done, hs->out), "cudaEventRecord");
    ATTN_HOST_CHECK(cudaStreamWaitEvent(caller, hs->done, 0), "cudaStreamWaitEvent");
#undef ATTN_HOST_CHECK
    return ATTN_OK;
}

ATTN_API attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o,
                                    float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                                    float descale_q, float descale_k, float descale_v,
                                    int mask_kind, int window, const int* seqlens_k,
                                    attn_stream_t stream) {
    bool nothing = false;
    attn_status_t st = check_fwd(q, k, v, o, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k,
                                 &nothing);
    if (st != ATTN_OK) return st;
    if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_fp8 supports d = 128 only (d=%d)", d);
    for (float f : {descale_q, descale_k, descale_v})
        if (!(f > 0.f) || !std::isfinite(f))
            return fail(ATTN_ERR_INVALID_ARG, "descale factors must be finite and > 0");
    if (!std::isfinite(scale * descale_q * descale_k * 1.4426950408889634f))
        return fail(ATTN_ERR_INVALID_ARG, "scale * descale_q * descale_k overflows FP32");
    if (nothing) return ATTN_OK;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = static_cast<long long>(B) * H * Nq;
    if (Nk == 0) {
        cudaError_t e = launch_fill_empty(o, lse, rows, d, true, s);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "fill kernel launch");
    }
    unsigned int* err = nullptr;
    if ((st = err_word(&err)) != ATTN_OK) return st;
    CUtensorMap tq, tk, tv, to;
    const long long bh = static_cast<long long>(B) * H;
    if ((st = encode_3d(&tq, q, d, Nq, bh, true)) != ATTN_OK) return st;
    if ((st = encode_3d(&tk, k, d, Nk, bh, true)) != ATTN_OK) return st;
    if ((st = encode_3d(&tv, v, d, Nk, bh, true)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&to, o, d, Nq, bh)) != ATTN_OK) return st;   // BF16 output
    FwdArgs a{q, k, v, o, lse, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k, err};
    cudaError_t e = launch_fwd_fp8_maps(a, descale_q, descale_k, descale_v, tq, tk, tv, to, s);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_fwd_fp8 kernel launch");
}

ATTN_API attn_status_t attn_fwd_f32(const float* q, const float* k, const float* v, float* o,
                                    float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                                    int mask_kind, int window, const int* seqlens_k,
                                    attn_stream_t stream) {
    bool nothing = false;
    attn_status_t st = check_fwd(q, k, v, o, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k,
                                 &nothing);
    if (st != ATTN_OK || nothing) return st;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = static_cast<long long>(B) * H * Nq;
    cudaError_t e;
    if (Nk == 0) {
        e = launch_fill_empty(o, lse, rows, d, false, s);
    } else {
        FwdArgs a{q, k, v, o, lse, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k, nullptr};
        e = launch_fwd_f32(a, s);
    }
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_fwd_f32 kernel launch");
}


ATTN_API size_t attn_decode_workspace_bytes(int B, int H, int d, int num_splits) {
    if (B < 0 || H < 0 || d <= 0 || num_splits < 1 || num_splits > 1024) return 0;
    const size_t slots = static_cast<size_t>(B) * H * num_splits;
    return align256(slots * d * sizeof(float)) + align256(slots * sizeof(float));
}

ATTN_API attn_status_t attn_decode_splitkv(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int B, int H, int Nk, int d, float scale,
                                           const int* seqlens_k, int num_splits, void* workspace,
                                           size_t workspace_bytes, attn_stream_t stream) {
    if (B < 0 || H < 0 || Nk < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d Nk=%d)", B, H, Nk);
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (num_splits < 1 || num_splits > 1024)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits=%d outside [1, 1024]", num_splits);
    if (B > 65535 || H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "B and H must be <= 65535");
    if (static_cast<long long>(B) * H == 0) return ATTN_OK;
    if (q == nullptr || o == nullptr) return fail(ATTN_ERR_INVALID_ARG, "q and o must not be NULL");
    if (Nk > 0 && (k == nullptr || v == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "k and v must not be NULL");
    if (!aligned16(q) || !aligned16(o) || (Nk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    const size_t need = attn_decode_workspace_bytes(B, H, d, num_splits);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need,
                    workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t slots = static_cast<size_t>(B) * H * num_splits;
    float* ws_o = static_cast<float*>(workspace);
    float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             align256(slots * d * sizeof(float)));
    DecodeArgs a{q, k, v, o, lse, B, H, Nk, d, scale, seqlens_k, num_splits, ws_o, ws_lse, nullptr};
    cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_decode_splitkv kernel launch");
}

ATTN_API attn_status_t attn_decode_splitkv_noalloc(const void* q, const void* k, const void* v,
                                                   void* o, float* lse, int B, int H, int Nk,
                                                   int d, float scale, const int* seqlens_k,
                                                   int num_splits, attn_stream_t stream) {
    if (B < 0 || H < 0 || Nk < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%d H=%d Nk=%d)", B, H, Nk);
    if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (num_splits < 1 || num_splits > 1024)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits=%d outside [1, 1024]", num_splits);
    if (B > 65535 || H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "B and H must be <= 65535");
    if (static_cast<long long>(B) * H == 0) return ATTN_OK;
    if (q == nullptr || o == nullptr) return fail(ATTN_ERR_INVALID_ARG, "q and o must not be NULL");
    if (Nk > 0 && (k == nullptr || v == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "k and v must not be NULL");
    if (!aligned16(q) || !aligned16(o) || (Nk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    const size_t need = attn_decode_workspace_bytes(B, H, d, num_splits);
    void* scratch = nullptr;
    size_t have = 0;
    cudaError_t e = decode_static_scratch(&scratch, &have);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    if (need > have)
        return fail(ATTN_ERR_INVALID_ARG,
                    "attn_decode_splitkv_noalloc: B*H*num_splits*(d+1) partials need %zu bytes, "
                    "more than the fixed %zu-byte scratch; use attn_decode_splitkv with a workspace",
                    need, have);
    const size_t slots = static_cast<size_t>(B) * H * num_splits;
    float* ws_o = static_cast<float*>(scratch);
    float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                             align256(slots * d * sizeof(float)));
    DecodeArgs a{q, k, v, o, lse, B, H, Nk, d, scale, seqlens_k, num_splits, ws_o, ws_lse, nullptr};
    e = launch_decode(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_decode_splitkv_noalloc kernel launch");
}

namespace {
size_t bwd_region(int B, int H, int Nq) {
    const size_t rows = static_cast<size_t>(B) * H * ((static_cast<size_t>(Nq) + 127) / 128 * 128);
    return align256(rows * sizeof(float));
}
}  // namespace

ATTN_API size_t attn_bwd_workspace_bytes(int B, int H, int Nq, int d) {
    if (B < 0 || H < 0 || Nq < 0 || (d != 64 && d != 128)) return 0;
    // lse and D rows; with dQ accumulated in the keys-outer kernel, an FP32
    // dQ accumulator of d values per (padded) query row after them
    return 2 * bwd_region(B, H, Nq) + (bwd_fused_dq(d) ? bwd_region(B, H, Nq) * d : 0);
}

ATTN_API attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int Nq, int Nk, int d, float scale, int mask_kind,
                                int window, const int* seqlens_k, void* workspace,
                                size_t workspace_bytes, attn_stream_t stream) {
    bool nothing = false;
    attn_status_t st = check_fwd(q, k, v, o, B, H, Nq, Nk, d, scale, mask_kind, window, seqlens_k,
                                 &nothing);
    if (st != ATTN_OK) return st;
    const long long bh = static_cast<long long>(B) * H;
    if (bh == 0) return ATTN_OK;
    if (Nq > 0 && (dout == nullptr || lse == nullptr || dq == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "dout, lse and dq must not be NULL");
    if (Nk > 0 && (dk == nullptr || dv == nullptr))
        return fail(ATTN_ERR_INVALID_ARG, "dk and dv must not be NULL");
    if ((Nq > 0 && (!aligned16(dout) || !aligned16(dq) ||
                    (reinterpret_cast<uintptr_t>(lse) & 3u))) ||
        (Nk > 0 && (!aligned16(dk) || !aligned16(dv))))
        return fail(ATTN_ERR_INVALID_ARG, "dout, dq, dk, dv must be 16-byte aligned, lse 4-byte");
    const size_t need = attn_bwd_workspace_bytes(B, H, Nq, d);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need,
                    workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (Nq == 0 || Nk == 0) {
        // no (query, key) pair: every gradient is zero
        if (Nq > 0 && (e = launch_fill_empty(dq, nullptr, bh * Nq, d, true, s)) != cudaSuccess)
            return cuda_fail(e, "fill kernel launch");
        if (Nk > 0) {
            if ((e = launch_fill_empty(dk, nullptr, bh * Nk, d, true, s)) != cudaSuccess ||
                (e = launch_fill_empty(dv, nullptr, bh * Nk, d, true, s)) != cudaSuccess)
                return cuda_fail(e, "fill kernel launch");
        }
        return ATTN_OK;
    }
    unsigned int* err = nullptr;
    if ((st = err_word(&err)) != ATTN_OK) return st;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tk64, tv64;
    if ((st = encode_bf16_3d(&tq, q, d, Nq, bh)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&tk, k, d, Nk, bh)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&tv, v, d, Nk, bh)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&tdo, dout, d, Nq, bh)) != ATTN_OK) return st;
    if ((st = encode_bf16_3d(&tdk, dk, d, Nk, bh)) != ATTN_OK) return st;   // the dK/dV stores
    if ((st = encode_bf16_3d(&tdv, dv, d, Nk, bh)) != ATTN_OK) return st;
    if ((st = encode_3d(&tk64, k, d, Nk, bh, false, 64)) != ATTN_OK) return st;   // dQ kernel units
    if ((st = encode_3d(&tv64, v, d, Nk, bh, false, 64)) != ATTN_OK) return st;
    float* ws_lse2 = static_cast<float*>(workspace);
    float* ws_dd = reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_region(B, H, Nq));
    float* ws_dq = bwd_fused_dq(d) ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                              2 * bwd_region(B, H, Nq))
                                   : nullptr;
    BwdArgs a{q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, mask_kind, window,
              seqlens_k, ws_lse2, ws_dd, ws_dq, err};
    e = launch_bwd(a, tq, tk, tv, tdo, tdk, tdv, tk64, tv64, s);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_bwd kernel launch");
}

ATTN_API attn_status_t attn_softmax_rows(const void* x, void* y, float* lse, long long rows,
                                         int n, int dtype, attn_stream_t stream) {
    if (rows < 0 || rows > 2147483647LL || n < 1)
        return fail(ATTN_ERR_INVALID_ARG, "rows must be in [0, 2^31), n >= 1 (rows=%lld n=%d)",
                    rows, n);
    if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16)
        return fail(ATTN_ERR_UNSUPPORTED, "dtype %d (ATTN_DTYPE_F32 or ATTN_DTYPE_BF16)", dtype);
    if (rows == 0) return ATTN_OK;
    if (x == nullptr || y == nullptr) return fail(ATTN_ERR_INVALID_ARG, "x and y must not be NULL");
    const size_t esz = dtype == ATTN_DTYPE_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & (esz - 1))
        return fail(ATTN_ERR_INVALID_ARG, "x and y must be aligned to their element size");
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    cudaError_t e = launch_softmax_rows(x, y, lse, rows, n, dtype == ATTN_DTYPE_BF16,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_softmax_rows kernel launch");
}

ATTN_API attn_status_t attn_check_device_error(attn_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int* word = nullptr;
    attn_status_t st = err_word(&word);
    if (st != ATTN_OK) return st;
    unsigned int w = 0;
    e = cudaMemcpy(&w, word, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    if (w != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear error word");
        return fail(ATTN_ERR_TIMEOUT, "device wait gave up (site %u)", w >> 8);
    }
    return ATTN_OK;
}

ATTN_API attn_status_t attn_exp2_soft(const float* x, float* y, long long n,
                                      attn_stream_t stream) {
    if (n < 0) return fail(ATTN_ERR_INVALID_ARG, "n must be >= 0");
    if (n == 0) return ATTN_OK;
    if (x == nullptr || y == nullptr) return fail(ATTN_ERR_INVALID_ARG, "x and y must not be NULL");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 3u)
        return fail(ATTN_ERR_INVALID_ARG, "x and y must be 4-byte aligned");
    const long long pairs = (n + 1) / 2;
    const unsigned grid = static_cast<unsigned>(std::min<long long>((pairs + 255) / 256, 4096));
    exp2_soft_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "attn_exp2_soft kernel launch");
}

ATTN_API attn_status_t attn_selftest_bounded_wait(long long limit_cycles, attn_stream_t stream) {
    if (limit_cycles < 1 || limit_cycles > (1LL << 31))
        return fail(ATTN_ERR_INVALID_ARG, "limit_cycles outside [1, 2^31]");
    unsigned int* err = nullptr;
    attn_status_t st = err_word(&err);
    if (st != ATTN_OK) return st;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_cycles);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "selftest kernel launch");
}

ATTN_API const char* attn_last_error(void) { return t_last_error.c_str(); }

ATTN_API const char* attn_version(void) { return "online_softmax_02_gb300 0.1.0 (sm_103a)"; }

namespace attn {
cudaError_t launch_fill_empty(void* o, float* lse, long long rows, int d, bool bf16,
                              cudaStream_t stream) {
    const long long n = rows * d;
    const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 4096));
    fill_empty_kernel<<<blocks, 256, 0, stream>>>(o, lse, rows, d, bf16 ? 1 : 0);
    return cudaGetLastError();
}
}  // namespace attn
