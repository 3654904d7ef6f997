// fwd_sm103.cu -- BF16 fused attention forward on the sm_103a tensor cores.
//
// The method is the query-tile online softmax of P2 ("Implement online
// softmax for a whole tile of queries, not one query, and write the rescaling
// step in matrix form", "A strong answer"): for a 128-row query tile Q_i and
// 128-key blocks K_j, V_j,
//   S_j = scale Q_i K_j^T,  m' = max(m, rowmax S_j),
//   m_ref = (m' == -inf ? 0 : m')            (the guard P2 gives for rows
//                                              that have not seen a key),
//   P_j = exp(S_j - m_ref),  alpha = exp(m - m_ref),
//   l' = alpha l + P_j 1,    A' = diag(alpha) A + P_j V_j,
// and O_i = diag(l)^-1 A once after the last block; lse = m + log l
// (P1 "Derive online softmax, prove it is exact, ...", "What interviewers
// probe next"). Blocks that the mask hides entirely are never loaded (P1
// "Common mistakes", on causal masking). The rescale of A is skipped for a
// warp whose 32 rows all kept their max (alpha is then exactly 1; P2 "What
// interviewers probe next").
//
// GB300 mapping (one CTA per SM, 320 threads):
//   * Two query tiles per CTA (256 rows) share every K/V block, so each
//     block is read from device memory once per 256 queries, and the tensor
//     core works on one tile's products while the other tile's softmax runs.
//   * Warp 8 issues TMA bulk-tensor loads: Q once, then K_j and V_j into a
//     2-stage ring of 128-byte-swizzled shared-memory buffers, tracked by
//     mbarriers with transaction counts.
//   * Warp 9 allocates 512 tensor-memory columns (S_0, S_1, O_0, O_1; FP32)
//     and one lane issues every tcgen05.mma: S_t = Q_t K_j^T with both
//     operands in shared memory, and O_t += P_t V_j with P_t read from tensor
//     memory (BF16, written over S_t) and V_j from shared memory. Issue order
//     per block: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j).
//   * Warps 0-3 run the softmax of tile 0 and warps 4-7 that of tile 1, one
//     thread per query row: tcgen05.ld of the 128 scores of its row, mask,
//     row max and row sum in registers (no shuffles: the row is in one
//     thread), exp2 with the scale folded into one FMA, P stored back to
//     tensor memory, A rescaled in tensor memory when a row's max moved, then
//     the epilogue O = A / l and lse.
//   * m, l and A are FP32; P is rounded to BF16 for the P V product.
//   * Every mbarrier wait is bounded; on expiry the CTA records the site in
//     the device error word, all roles stop, in-flight copies and MMAs are
//     drained, tensor memory is freed and the kernel returns.
#include <climits>
#include "common.cuh"

namespace attn {
namespace {

constexpr int BM = 128;                 // query rows per tile
constexpr int NT = 2;                   // query tiles per CTA
constexpr int BN = 128;                 // keys per block
constexpr int kSoftmaxWarps = 4 * NT;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
    static constexpr int kStages = (D == 64) ? 4 : 2;
    static constexpr uint32_t kRowBytes = 128;                 // one swizzle atom row
    static constexpr uint32_t kQTileBytes = BM * D * 2;
    static constexpr uint32_t kKVBytes = BN * D * 2;
    static constexpr uint32_t kQChunkBytes = BM * kRowBytes;   // 64 head dims of a Q tile
    static constexpr uint32_t kKVChunkBytes = BN * kRowBytes;  // 64 head dims of a K/V block
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKOff = kQOff + NT * kQTileBytes;
    static constexpr uint32_t kVOff = kKOff + kStages * kKVBytes;
    static constexpr uint32_t kBarOff = kVOff + kStages * kKVBytes;
    // barrier indices
    static constexpr int bQFull = 0;
    static constexpr int bKFull = 1;
    static constexpr int bKEmpty = bKFull + kStages;
    static constexpr int bVFull = bKEmpty + kStages;
    static constexpr int bVEmpty = bVFull + kStages;
    static constexpr int bSFull = bVEmpty + kStages;
    static constexpr int bPFull = bSFull + NT;
    static constexpr int bODone = bPFull + NT;
    static constexpr int bDrain = bODone + NT;
    static constexpr int kNumBars = bDrain + 1;
    static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag
    static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
    static constexpr uint32_t s_col(int t) { return t * BN; }
    static constexpr uint32_t o_col(int t) { return NT * BN + t * D; }
    static_assert(NT * BN + NT * D <= kTmemCols, "tensor memory budget");
};

struct Range { int lo, hi; };   // key blocks [lo, hi)

// Key blocks that some row of the tile [row_first, row_first + BM) can see.
__device__ __forceinline__ Range tile_range(int row_first, int Nq, int Lk, bool causal,
                                            bool windowed, int window) {
    if (row_first >= Nq) return {0, 0};
    const int row_last = min(row_first + BM, Nq) - 1;
    int key_hi = Lk;
    if (causal) key_hi = min(key_hi, row_last + 1);
    const int key_lo = windowed ? max(0, row_first - window + 1) : 0;
    if (key_lo >= key_hi) return {0, 0};
    return {key_lo / BN, (key_hi + BN - 1) / BN};
}

// True when some (row, key) pair of the block is hidden, so the softmax has
// to test keys one by one.
__device__ __forceinline__ bool block_needs_mask(int kb, int row_first, int Lk, bool causal,
                                                 bool windowed, int window) {
    const int ke = kb + BN;
    if (ke > Lk) return true;
    if (causal && ke - 1 > row_first) return true;
    if (windowed && kb <= row_first + BM - 1 - window) return true;
    return false;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ lse, int H, int Nq, int Nk, float scale_log2, int mask_kind,
                 int window, const int* __restrict__ seqlens_k, unsigned int* __restrict__ err,
                 int reverse_order) {
    using C = Cfg<D>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int pair = reverse_order ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * H + h;
    const int q0 = pair * (BM * NT);

    int Lk = Nk;
    if (mask_kind & kMaskPadding) Lk = min(max(seqlens_k[b], 0), Nk);
    const bool causal = (mask_kind & (kMaskCausal | kMaskWindow)) != 0;
    const bool windowed = (mask_kind & kMaskWindow) != 0;

    Range R[NT];
    int lo = INT_MAX, hi = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        R[t] = tile_range(q0 + t * BM, Nq, Lk, causal, windowed, window);
        if (R[t].lo < R[t].hi) { lo = min(lo, R[t].lo); hi = max(hi, R[t].hi); }
    }
    if (hi == 0) lo = 0;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(C::bQFull), 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar(C::bKFull + s), 1);
            ptx::mbar_init(bar(C::bKEmpty + s), 1);
            ptx::mbar_init(bar(C::bVFull + s), 1);
            ptx::mbar_init(bar(C::bVEmpty + s), 1);
        }
        for (int t = 0; t < NT; ++t) {
            ptx::mbar_init(bar(C::bSFull + t), 1);
            ptx::mbar_init(bar(C::bPFull + t), 4);   // one arrival per softmax warp
            ptx::mbar_init(bar(C::bODone + t), 1);
        }
        ptx::mbar_init(bar(C::bDrain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && lo < hi) {
            ptx::prefetch_tmap(&tm_q);
            ptx::prefetch_tmap(&tm_k);
            ptx::prefetch_tmap(&tm_v);
            ptx::mbar_arrive_expect_tx(bar(C::bQFull), NT * C::kQTileBytes);
            for (int t = 0; t < NT; ++t)
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(sbase + C::kQOff + t * C::kQTileBytes + c * C::kQChunkBytes,
                                     &tm_q, bar(C::bQFull), c * 64, q0 + t * BM, bh);
            int issued = 0;
            for (int s = lo; s < hi; ++s) {
                const int i = s - lo, st = i % NS;
                const uint32_t ph = (i / NS) & 1;
                if (!wait_bounded(bar(C::bKEmpty + st), ph ^ 1, abort_flag, err, kSiteKEmpty)) break;
                ptx::mbar_arrive_expect_tx(bar(C::bKFull + st), C::kKVBytes);
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(sbase + C::kKOff + st * C::kKVBytes + c * C::kKVChunkBytes,
                                     &tm_k, bar(C::bKFull + st), c * 64, s * BN, bh);
                if (!wait_bounded(bar(C::bVEmpty + st), ph ^ 1, abort_flag, err, kSiteVEmpty)) {
                    issued = 2 * i + 1;
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(C::bVFull + st), C::kKVBytes);
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(sbase + C::kVOff + st * C::kKVBytes + c * C::kKVChunkBytes,
                                     &tm_v, bar(C::bVFull + st), c * 64, s * BN, bh);
                issued = 2 * (i + 1);
            }
            if (*abort_flag) {
                // Let the copies this thread started land before the CTA exits.
                wait_bounded(bar(C::bQFull), 0, nullptr, err, kSiteDrain, kWaitLimitCycles / 8);
                for (int n = max(0, issued - 2 * NS); n < issued; ++n) {
                    const int i = n / 2, st = i % NS;
                    const uint32_t ph = (i / NS) & 1;
                    wait_bounded(bar(((n & 1) ? C::bVFull : C::bKFull) + st), ph, nullptr, err,
                                 kSiteDrain, kWaitLimitCycles / 8);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && lo < hi) {
            constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(BM, D, true);
            int p_seen[NT], pv_done[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) { p_seen[t] = 0; pv_done[t] = 0; }
            bool ok = wait_bounded(bar(C::bQFull), 0, abort_flag, err, kSiteQFull);
            for (int s = lo; ok && s <= hi; ++s) {
                const int i = s - lo, st = i % NS;
                const uint32_t ph = (i / NS) & 1;
                const int pst = (i + NS - 1) % NS;
                const uint32_t pph = ((i - 1) / NS) & 1;
                if (s - 1 >= lo) {
                    ok = wait_bounded(bar(C::bVFull + pst), pph, abort_flag, err, kSiteVFull);
                    if (!ok) break;
                }
                if (s < hi) {
                    ok = wait_bounded(bar(C::bKFull + st), ph, abort_flag, err, kSiteKFull);
                    if (!ok) break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (s - 1 >= R[t].lo && s - 1 < R[t].hi) {
                        // O_t (+)= P_t V_{s-1}
                        ok = wait_bounded(bar(C::bPFull + t), p_seen[t] & 1, abort_flag, err,
                                          kSitePFull);
                        if (!ok) break;
                        ++p_seen[t];
                        ptx::tc_fence_after();
                        const uint32_t vbase = sbase + C::kVOff + pst * C::kKVBytes;
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            const uint64_t bdesc =
                                ptx::sdesc_sw128(vbase + kk * 16 * C::kRowBytes, C::kKVChunkBytes, 1024);
                            ptx::mma_ts(tmem + C::o_col(t), tmem + C::s_col(t) + kk * 8, bdesc,
                                        kIdescPV, (pv_done[t] > 0 || kk > 0) ? 1u : 0u);
                        }
                        ++pv_done[t];
                        if (s - 1 == R[t].hi - 1) ptx::mma_commit(bar(C::bODone + t));
                    }
                    if (s < hi && s >= R[t].lo && s < R[t].hi) {
                        // S_t = Q_t K_s^T
                        const uint32_t qbase = sbase + C::kQOff + t * C::kQTileBytes;
                        const uint32_t kbase = sbase + C::kKOff + st * C::kKVBytes;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t koff = (kk / 4) * C::kQChunkBytes + (kk % 4) * 32;
                            const uint32_t boff = (kk / 4) * C::kKVChunkBytes + (kk % 4) * 32;
                            const uint64_t adesc = ptx::sdesc_sw128(qbase + koff, 16, 1024);
                            const uint64_t bdesc = ptx::sdesc_sw128(kbase + boff, 16, 1024);
                            ptx::mma_ss(tmem + C::s_col(t), adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
                        }
                        ptx::mma_commit(bar(C::bSFull + t));
                    }
                }
                if (!ok) break;
                if (s - 1 >= lo) ptx::mma_commit(bar(C::bVEmpty + pst));
                if (s < hi) ptx::mma_commit(bar(C::bKEmpty + st));
            }
            // Every MMA issued above completes before tensor memory is freed.
            ptx::mma_commit(bar(C::bDrain));
            wait_bounded(bar(C::bDrain), 0, nullptr, err, kSiteDrain);
        }
    } else {
        // ------------------------------------------------ softmax, epilogue
        const int t = warp / 4, wq = warp % 4;
        const int r = wq * 32 + lane;
        const int row = q0 + t * BM + r;
        const int row_first = q0 + t * BM;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + C::s_col(t);
        const uint32_t o_addr = tmem + lane_base + C::o_col(t);
        float m = -INFINITY, l = 0.f;
        int c = 0;
        bool ok = true;
        for (int j = R[t].lo; j < R[t].hi; ++j, ++c) {
            const bool got = wait_bounded(bar(C::bSFull + t), c & 1, abort_flag, err, kSiteSFull);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            ptx::tc_fence_after();
            uint32_t sr[BN];
            ptx::tmem_ld32x32b_x128(s_addr, sr);
            const int kb = j * BN;
            if (block_needs_mask(kb, row_first, Lk, causal, windowed, window)) {
#pragma unroll
                for (int kk = 0; kk < BN; ++kk) {
                    const int key = kb + kk;
                    bool vis = key < Lk;
                    if (causal) vis = vis && key <= row;
                    if (windowed) vis = vis && key > row - window;
                    if (!vis) sr[kk] = __float_as_uint(-INFINITY);
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int kk = 0; kk < BN; ++kk) mx = fmaxf(mx, __uint_as_float(sr[kk]));
            const float m_new = fmaxf(m, mx * scale_log2);
            const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
            float sum = 0.f;
            uint32_t pk[BN / 2];
#pragma unroll
            for (int kk = 0; kk < BN / 2; ++kk) {
                const float p0 = ptx::ex2(fmaf(__uint_as_float(sr[2 * kk]), scale_log2, -m_ref));
                const float p1 = ptx::ex2(fmaf(__uint_as_float(sr[2 * kk + 1]), scale_log2, -m_ref));
                sum += p0 + p1;
                pk[kk] = pack_bf16x2(p0, p1);
            }
            ptx::tmem_st32x32b_x64(s_addr, pk);
            const float alpha = ptx::ex2(m - m_ref);
            l = fmaf(l, alpha, sum);
            const bool need = (m_new != m) && (m != -INFINITY);
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    ptx::tmem_ld32x32b_x32(o_addr + cc * 32, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    ptx::tmem_st32x32b_x32(o_addr + cc * 32, ov);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::bPFull + t));
            m = m_new;
        }
        if (ok && c > 0) {
            const bool got = wait_bounded(bar(C::bODone + t), 0, abort_flag, err, kSiteODone);
            ok = __all_sync(0xffffffffu, got);
            ptx::tc_fence_after();
        }
        const bool have = ok && c > 0;
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        __nv_bfloat16* orow = o + (static_cast<long long>(bh) * Nq + row) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            if (have) {
                ptx::tmem_ld32x32b_x32(o_addr + cc * 32, ov);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = 0u;
            }
            if (row < Nq) {
                uint32_t pw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pw[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l,
                                        __uint_as_float(ov[2 * e + 1]) * inv_l);
                uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(pw[4 * e], pw[4 * e + 1], pw[4 * e + 2], pw[4 * e + 3]);
            }
        }
        if (lse != nullptr && row < Nq)
            lse[static_cast<long long>(bh) * Nq + row] =
                (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t stream) {
    using C = Cfg<D>;
    static int configured_device = -1;   // attribute is per device; set once per device seen
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(fwd_sm103_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int pairs = (a.Nq + BM * NT - 1) / (BM * NT);
    dim3 grid(pairs, a.H, a.B);
    const int reverse = (a.mask_kind & (kMaskCausal | kMaskWindow)) ? 1 : 0;
    fwd_sm103_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(
        tq, tk, tv, static_cast<__nv_bfloat16*>(a.o), a.lse, a.H, a.Nq, a.Nk, a.scale * kLog2e,
        a.mask_kind, a.window, a.seqlens_k, a.err, reverse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_sm103_maps(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, cudaStream_t stream) {
    return a.d == 64 ? launch_d<64>(a, tq, tk, tv, stream) : launch_d<128>(a, tq, tk, tv, stream);
}

}  // namespace attn
