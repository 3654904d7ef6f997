// softmax.cu -- standalone row softmax with the online normalizer.
//
// P3 ("Online softmax", interview.clozo.ai): "Step 2" reads a vector once and
// keeps the pair (m, l) -- the running maximum and the sum of exp(x - m),
// the sum multiplied by exp(m_old - m_new) whenever the maximum grows;
// "Step 3" turns the final pair into outputs exp(x_i - m) / l in a second
// pass; "Step 4" merges pairs of different blocks with the same rescaling,
// which is associative, so a row can be split across threads, warps, CTAs.
// The table in "Trade-offs and edge cases" counts three memory accesses per
// element for this two-pass form (two reads, one write) against four for
// safe softmax.
//
// GB300 mapping. Every thread streams 16-byte vectors and keeps its own pair,
// updated once per vector (one exp per element plus one per vector). Four
// shapes by row length (in 16-byte vectors: 4 FP32 or 8 BF16 values):
//   warp mode     up to 512 vectors: one warp per row, 8 rows per CTA, the
//                 row held in registers, pairs merged by shuffles only;
//   CTA mode      up to 2048 vectors: one 256-thread CTA per row, the row in
//                 registers (HBM sees one read and one write per element),
//                 pairs merged by shuffles and shared memory; small enough
//                 that three CTAs share an SM and overlap load and store
//                 phases;
//   streamed      up to 8192 vectors: a 512-thread CTA per row reads the row
//                 twice with eight loads in flight per thread; the second
//                 read is served by L2 (the concurrent rows fit in it);
//   cluster       longer rows: a cluster of up to 8 streamed CTAs splits the
//                 row so that each slice stays L2-sized, and the CTA pairs
//                 meet through distributed shared memory.
// Measured alternatives on GB300: holding long rows in registers across a
// cluster (the cluster barrier and co-scheduling cost more than the saved
// L2 re-read), and a persistent CTA that holds row r in registers while a
// bulk copy brings row r+1 into shared memory (one row per SM in flight is
// too little).
// Rows whose length is not a multiple of the vector width, or whose base is
// not 16-byte aligned, take a one-element-per-load CTA kernel.
// In place (y == x) is allowed: every element is written by the thread that
// read it, after the row's pair is complete, and nothing reads x through the
// non-coherent path (x and y are not declared restrict).
#include "common.cuh"

namespace attn {
namespace {

constexpr int kCtaThreads = 256;        // register-held CTA mode, scalar kernel
constexpr int kWarpRowsPerCta = 8;      // warp mode: 8 warps, one row each
constexpr int kWarpKeepMax = 16;        // warp mode: vectors per lane
constexpr int kCtaKeep = 8;             // CTA mode: vectors per thread
constexpr int kStreamThreads = 512;     // streamed mode
constexpr int kStreamUnroll = 8;        // streamed mode: loads in flight per thread
constexpr int kStreamSlice = 8192;      // streamed mode: vectors per CTA before splitting
constexpr int kMaxCluster = 8;          // portable cluster size
constexpr float kLog2eS = 1.4426950408889634f;
constexpr float kLn2S = 0.6931471805599453f;

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void to_f32(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 from_f32(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static float one(const float* p) { return *p; }
    __device__ static void store_one(float* p, float v) { *p = v; }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_f32(const uint4& u, float* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { f[2 * i] = bf16lo_to_f32(w[i]); f[2 * i + 1] = bf16hi_to_f32(w[i]); }
    }
    __device__ static uint4 from_f32(const float* f) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
    __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    __device__ static void store_one(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// Pair (m, l) in log2 units: m = max x*log2(e), l = sum exp2(x*log2(e) - m).
struct Pair { float m, l; };

// P3 "Step 4": the merged max is the larger; each sum is rescaled to it.
__device__ __forceinline__ Pair merge(Pair a, Pair b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {-INFINITY, 0.f};
    return {m, a.l * ptx::ex2(a.m - m) + b.l * ptx::ex2(b.m - m)};
}

// P3 "Step 2" for one vector of values: new max, old sum rescaled, new terms.
template <int N>
__device__ __forceinline__ Pair update(Pair p, const float* f) {
    float vm = f[0];
#pragma unroll
    for (int i = 1; i < N; ++i) vm = fmaxf(vm, f[i]);
    const float m_new = fmaxf(p.m, vm * kLog2eS);
    if (m_new == -INFINITY) return p;                  // nothing finite seen yet
    float l = p.l * ptx::ex2(p.m - m_new);
#pragma unroll
    for (int i = 0; i < N; ++i) l += ptx::ex2(fmaf(f[i], kLog2eS, -m_new));
    return {m_new, l};
}

// Butterfly over the 32 lanes: every lane ends with the warp's pair.
__device__ __forceinline__ Pair warp_merge(Pair p) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        Pair o;
        o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
        o.l = __shfl_xor_sync(0xffffffffu, p.l, off);
        p = merge(p, o);
    }
    return p;
}

// Warps, then the per-warp pairs (at most 32 warps): every thread gets the CTA's pair.
__device__ __forceinline__ Pair cta_merge(Pair p, Pair* red) {
    p = warp_merge(p);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) red[warp] = p;
    __syncthreads();
    const int nw = (blockDim.x + 31) / 32;
    return warp_merge((lane < nw) ? red[lane] : Pair{-INFINITY, 0.f});
}

// Output of one vector: exp2(x*log2e - m) / l, computed as a product with 1/l.
template <typename T>
__device__ __forceinline__ uint4 normalize(const uint4& u, float mref, float inv) {
    using V = Vec<T>;
    float f[V::N];
    V::to_f32(u, f);
#pragma unroll
    for (int i = 0; i < V::N; ++i) f[i] = ptx::ex2(fmaf(f[i], kLog2eS, -mref)) * inv;
    return V::from_f32(f);
}

__device__ __forceinline__ void finish(const Pair& tot, float* mref, float* inv) {
    *inv = (tot.l > 0.f) ? 1.f / tot.l : 0.f;          // all -inf: outputs 0
    *mref = (tot.m == -INFINITY) ? 0.f : tot.m;
}

__device__ __forceinline__ float row_lse(const Pair& tot) {
    return (tot.l > 0.f) ? (tot.m + log2f(tot.l)) * kLn2S : -INFINITY;
}

// Warp mode: one warp per row, R vectors per lane kept in registers.
template <typename T, int R>
__global__ void __launch_bounds__(kWarpRowsPerCta * 32)
softmax_rows_warp_kernel(const T* x, T* y, float* __restrict__ lse,
                         long long rows, int n) {
    using V = Vec<T>;
    const int lane = threadIdx.x % 32;
    const long long row = static_cast<long long>(blockIdx.x) * kWarpRowsPerCta + threadIdx.x / 32;
    if (row >= rows) return;                           // whole warp leaves together
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * n);
    uint4* yr = reinterpret_cast<uint4*>(y + row * n);
    const int nvec = n / V::N;
    uint4 keep[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int iv = lane + 32 * r;
        keep[r] = (iv < nvec) ? __ldcs(xr + iv) : make_uint4(0, 0, 0, 0);
    }
    Pair p{-INFINITY, 0.f};
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (lane + 32 * r < nvec) {
            float f[V::N];
            V::to_f32(keep[r], f);
            p = update<V::N>(p, f);
        }
    }
    const Pair tot = warp_merge(p);
    float mref, inv;
    finish(tot, &mref, &inv);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int iv = lane + 32 * r;
        if (iv < nvec) __stcs(yr + iv, normalize<T>(keep[r], mref, inv));
    }
    if (lse != nullptr && lane == 0) lse[row] = row_lse(tot);
}

// CTA / cluster mode: the row is split over the `csize` CTAs of a cluster
// (csize = 1: a plain CTA per row); CTA `rank` owns the contiguous slice
// [rank*S, min(nvec, (rank+1)*S)) of vectors, S = ceil(nvec / csize).
// R > 0: the slice (at most R vectors per thread) stays in registers.
// R = 0: the slice is read twice, kStreamUnroll independent 16-byte loads in
// flight per thread; the second pass walks the slice from its end, so it
// starts with the lines the first pass loaded last (the likeliest to still be
// in L2).
template <typename T, int THREADS, int R>
__global__ void __launch_bounds__(THREADS, R > 0 ? 3 : 2)
softmax_rows_cta_kernel(const T* x, T* y, float* __restrict__ lse,
                        int n, int csize) {
    using V = Vec<T>;
    constexpr int U = kStreamUnroll;
    __shared__ Pair red[THREADS / 32];
    __shared__ float2 cta_pair;
    const int rank = csize > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
    const long long row = blockIdx.x / csize;
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * n);
    uint4* yr = reinterpret_cast<uint4*>(y + row * n);
    const int nvec = n / V::N;
    const int S = (nvec + csize - 1) / csize;
    const int lo = rank * S;
    const int hi = min(nvec, lo + S);
    const int tid = threadIdx.x;
    Pair p{-INFINITY, 0.f};
    uint4 keep[R > 0 ? R : 1];
    if (R > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int iv = lo + tid + r * THREADS;
            keep[r] = (iv < hi) ? __ldcs(xr + iv) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (lo + tid + r * THREADS < hi) {
                float f[V::N];
                V::to_f32(keep[r], f);
                p = update<V::N>(p, f);
            }
        }
    } else {
        int iv = lo + tid;
        for (; iv + (U - 1) * THREADS < hi; iv += U * THREADS) {
            uint4 a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = xr[iv + u * THREADS];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float f[V::N];
                V::to_f32(a[u], f);
                p = update<V::N>(p, f);
            }
        }
        for (; iv < hi; iv += THREADS) {
            float f[V::N];
            V::to_f32(xr[iv], f);
            p = update<V::N>(p, f);
        }
    }
    Pair tot = cta_merge(p, red);
    if (csize > 1) {
        // Publish this CTA's pair, then merge all csize pairs in rank order
        // (every CTA of the cluster gets the same row pair).
        if (tid == 0) cta_pair = make_float2(tot.m, tot.l);
        ptx::cluster_arrive_release();
        ptx::cluster_wait_acquire();
        const uint32_t mine = ptx::smem_u32(&cta_pair);
        Pair all{-INFINITY, 0.f};
        for (int r = 0; r < csize; ++r) {
            const float2 v = ptx::ld_dsmem_f32x2(ptx::mapa_shared(mine, r));
            all = merge(all, Pair{v.x, v.y});
        }
        tot = all;
        ptx::cluster_arrive_release();     // this CTA is done reading its peers
    }
    float mref, inv;
    finish(tot, &mref, &inv);
    if (R > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int iv = lo + tid + r * THREADS;
            if (iv < hi) __stcs(yr + iv, normalize<T>(keep[r], mref, inv));
        }
    } else {
        int jv = hi - 1 - tid;
        for (; jv - (U - 1) * THREADS >= lo; jv -= U * THREADS) {
            uint4 a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = __ldcs(xr + jv - u * THREADS);
#pragma unroll
            for (int u = 0; u < U; ++u) __stcs(yr + jv - u * THREADS, normalize<T>(a[u], mref, inv));
        }
        for (; jv >= lo; jv -= THREADS) __stcs(yr + jv, normalize<T>(__ldcs(xr + jv), mref, inv));
    }
    if (lse != nullptr && rank == 0 && tid == 0) lse[row] = row_lse(tot);
    if (csize > 1) ptx::cluster_wait_acquire();   // peers may still read cta_pair
}

// Any row length / alignment: element by element (same two passes).
template <typename T>
__global__ void __launch_bounds__(kCtaThreads)
softmax_rows_scalar_kernel(const T* x, T* y, float* __restrict__ lse,
                           int n) {
    using V = Vec<T>;
    __shared__ Pair red[kCtaThreads / 32];
    const long long row = blockIdx.x;
    const T* xr = x + row * n;
    T* yr = y + row * n;
    Pair p{-INFINITY, 0.f};
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float f = V::one(xr + i);
        p = update<1>(p, &f);
    }
    const Pair tot = cta_merge(p, red);
    float mref, inv;
    finish(tot, &mref, &inv);
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        V::store_one(yr + i, ptx::ex2(fmaf(V::one(xr + i), kLog2eS, -mref)) * inv);
    if (lse != nullptr && threadIdx.x == 0) lse[row] = row_lse(tot);
}

template <typename T, int R>
cudaError_t launch_warp(const T* x, T* y, float* lse, long long rows, int n, cudaStream_t st) {
    const long long grid = (rows + kWarpRowsPerCta - 1) / kWarpRowsPerCta;
    softmax_rows_warp_kernel<T, R><<<static_cast<unsigned>(grid), kWarpRowsPerCta * 32, 0, st>>>(
        x, y, lse, rows, n);
    return cudaGetLastError();
}

template <typename T, int THREADS, int R>
cudaError_t launch_cta(const T* x, T* y, float* lse, long long rows, int n, int csize,
                       cudaStream_t st) {
    const long long grid = rows * csize;
    if (grid > 2147483647LL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = csize > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, softmax_rows_cta_kernel<T, THREADS, R>, x, y, lse, n, csize);
}

template <typename T>
cudaError_t launch_t(const void* xv, void* yv, float* lse, long long rows, int n,
                     cudaStream_t st) {
    using V = Vec<T>;
    const T* x = static_cast<const T*>(xv);
    T* y = static_cast<T*>(yv);
    const bool vec_ok = (n % V::N == 0) && ((reinterpret_cast<uintptr_t>(xv) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(yv) & 15u) == 0);
    if (!vec_ok) {
        if (rows > 2147483647LL) return cudaErrorInvalidConfiguration;
        softmax_rows_scalar_kernel<T><<<static_cast<unsigned>(rows), kCtaThreads, 0, st>>>(
            x, y, lse, n);
        return cudaGetLastError();
    }
    const int nvec = n / V::N;
    if (nvec <= 32 * kWarpKeepMax) {                   // warp mode
        const int per = (nvec + 31) / 32;
        if (per <= 1) return launch_warp<T, 1>(x, y, lse, rows, n, st);
        if (per <= 2) return launch_warp<T, 2>(x, y, lse, rows, n, st);
        if (per <= 4) return launch_warp<T, 4>(x, y, lse, rows, n, st);
        if (per <= 8) return launch_warp<T, 8>(x, y, lse, rows, n, st);
        return launch_warp<T, kWarpKeepMax>(x, y, lse, rows, n, st);
    }
    if (nvec <= kCtaThreads * 4) return launch_cta<T, kCtaThreads, 4>(x, y, lse, rows, n, 1, st);
    if (nvec <= kCtaThreads * kCtaKeep)
        return launch_cta<T, kCtaThreads, kCtaKeep>(x, y, lse, rows, n, 1, st);
    // Streamed slices of at most kStreamSlice vectors, one CTA per slice.
    const int csize = min(kMaxCluster, (nvec + kStreamSlice - 1) / kStreamSlice);
    return launch_cta<T, kStreamThreads, 0>(x, y, lse, rows, n, csize, st);
}

}  // namespace

cudaError_t launch_softmax_rows(const void* x, void* y, float* lse, long long rows, int n,
                                bool bf16, cudaStream_t stream) {
    return bf16 ? launch_t<__nv_bfloat16>(x, y, lse, rows, n, stream)
                : launch_t<float>(x, y, lse, rows, n, stream);
}

}  // namespace attn
