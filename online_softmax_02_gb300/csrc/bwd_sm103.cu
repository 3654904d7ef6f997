// bwd_sm103.cu -- attention backward on the sm_103a tensor cores.
//
// The forward pass keeps only O and the per-row log-sum-exp (P1 "Derive
// online softmax, prove it is exact, ...", "What interviewers probe next":
// the backward kernel recomputes P block by block from Q, K and that
// scalar); the backward rebuilds the normalised P_j = exp(S_j - LSE)
// directly, with no running max (P2 "Implement online softmax for a whole
// tile of queries ...", closing paragraph on the backward pass). With
// D_i = sum_t dO_it O_it, the gradients are
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches (d = 128):
//   bwd_prep_kernel   D_i and LSE_i * log2(e) per query row into the
//                     workspace, rows padded to a multiple of 128 (padding
//                     rows get LSE = +inf, D = 0, so they contribute P = 0);
//                     zeroes the FP32 dQ accumulator.
//   bwd_dkdv_kernel   keys outer: a CTA owns 128 keys of one (b, h) and walks
//                     the query blocks in units of 64 queries. Per unit:
//                     S^T = K Q_u^T and dP^T = V dO_u^T (M = 128 keys, N = 64)
//                     into one of two tensor-memory buffers; one thread per
//                     key row turns them into P^T and dS^T (BF16, written back
//                     into the buffer, dS^T also into shared memory); then
//                     dQ_u^T = K^T dS_u^T (M = d, N = 64: the unit's dQ,
//                     transposed, into the buffer's dP^T columns, which are
//                     read by then), dV += P^T dO_u and dK += dS^T Q_u
//                     (A operand from TMEM) accumulate in tensor memory. Four
//                     dQ warps read dQ_u^T out and add it into the FP32
//                     accumulator with red.global.add (one 128-byte line per
//                     warp instruction). Five products per unit, none
//                     recomputed. At the end dK and dV leave through the
//                     CTA's K and V tiles by TMA stores.
//   bwd_dq_convert_kernel  dQ = scale * accumulator, rounded to BF16.
// d = 64 (and builds with ATTN_BWD_FUSED_DQ=0) keep dQ in its own pass:
//   bwd_dq_kernel     queries outer: a CTA owns 128 queries; per unit of 64
//                     keys S = Q K_u^T, dP = dO V_u^T, dS (BF16, TMEM), and
//                     dQ += dS K_u in tensor memory (S and dP computed twice:
//                     seven products per unit pair instead of five).
// On the prefill shape (B1 H64 8192^2 d128) the fused form measures 4.92 ms
// per step against 5.53 ms: the dQ reductions (17 GB of FP32 partial sums
// per step, into an accumulator that stays in L2 while a head's CTAs run)
// cost about 0.9 ms of the 1.9 ms that dropping the two recomputed products
// saves. The reduction order of dQ across key blocks is not fixed, so dQ may
// differ in its last bit from run to run; dK and dV are reproducible.
//
// Pipelining. Two unit buffers in tensor memory per kernel (in the dQ
// kernel K and V arrive as 64-key units in a ring of six slots, which the
// row warps release; Q and dO sit in tensor memory as the A operand of the
// score products) let the MMA warp issue the next unit's products while
// the row warps work; S and dP are committed separately, so the row warps
// compute P as soon as S is done (while dP's product runs); in the dK/dV
// kernel dV's and dK's products are issued together once dS^T is stored
// (one wait in the issue stream instead of two: 5.66 -> 5.60 ms). Row work
// goes 32 columns at a time with the block's LSE and D read as 16-byte
// shared-memory vectors. Both MMA loops are peeled so that their bodies
// hold no tests beyond the waits.
// Measured on GB300 (B1 H64 8192^2 d128): with the element-wise work taken
// out the two kernels are only 8 % faster, so the limit is the MMA issue
// stream itself (waits between the single issuer's groups drain the short
// tensor queue), not the softmax.
//
// Warp roles (192 threads with 4 row warps): the row warps hold one thread
// per row (TMEM lanes 0-127), then the TMA producer warp and the MMA issuer /
// TMEM owner warp; those two run their loops on the whole warp and issue
// from one elected lane. Every wait is bounded.
#include <algorithm>
#include <climits>
#include "common.cuh"

namespace attn {
namespace {

constexpr int BT = 128;                   // rows per tile (queries or keys)
constexpr int BU = 64;                    // rows of the inner tile per pipeline unit
// Row warps: 4 (one per TMEM lane quarter; measured fastest) or 8 (two per
// quarter, each taking half of a unit's columns: 6 % slower, the eight
// arrivals per hand-off cost more than the shorter row work saves).
#ifndef ATTN_BWD_ROW_WARPS
#define ATTN_BWD_ROW_WARPS 4
#endif
constexpr int kRowWarpsB = ATTN_BWD_ROW_WARPS;
static_assert(kRowWarpsB == 4 || kRowWarpsB == 8, "4 or 8 row warps");
constexpr int kQuartersPerWarp = (BU / 32) / (kRowWarpsB / 4);
constexpr int kThreadsB = (kRowWarpsB + 2) * 32;
constexpr int kProdWarp = kRowWarpsB, kMmaWarpB = kRowWarpsB + 1;
constexpr int NSB = 2;                    // ring stages
constexpr uint32_t kTmemColsB = 512;
constexpr float kLog2eB = 1.4426950408889634f;

// Column (within a unit buffer) of the BF16 operand for K-step kk (16 rows
// of the unit's inner dimension): each row warp writes its 32 rows' packed
// values (16 columns) at the start of its own 32 score columns, so the two
// warps that share a lane quarter never write columns the other still reads.
__host__ __device__ constexpr uint32_t a_col(int kk) { return (kk / 2) * 32 + (kk % 2) * 8; }

template <int D>
struct BCfg {
    static constexpr uint32_t kRowBytes = 128;
    static constexpr uint32_t kTileBytes = BT * D * 2;          // one 128-row tile
    static constexpr uint32_t kChunkBytes = BT * kRowBytes;     // 64 head dims of a tile
    static constexpr uint32_t kUnitBytes = BU * kRowBytes;      // offset of the second half
};

// --- dK/dV kernel shared memory: K, V once; ring of {Q, dO, LSE2, D};
// with FQ (dQ accumulated here) also the unit's dS^T as the B operand of
// dQ^T = K^T dS^T ---
template <int D, bool FQ = false>
struct KVCfg : BCfg<D> {
    using B = BCfg<D>;
    static constexpr uint32_t kKOff = 0;
    static constexpr uint32_t kVOff = B::kTileBytes;
    static constexpr uint32_t kRowVals = 2 * BT * 4;           // the rows' LSE and D
    static constexpr uint32_t kStageBytes = 2 * B::kTileBytes + kRowVals;
    static constexpr uint32_t kRingOff = 2 * B::kTileBytes;
    static constexpr uint32_t q_off(int s) { return kRingOff + s * kStageBytes; }
    static constexpr uint32_t do_off(int s) { return q_off(s) + B::kTileBytes; }
    static constexpr uint32_t lse_off(int s) { return q_off(s) + 2 * B::kTileBytes; }
    static constexpr uint32_t dd_off(int s) { return lse_off(s) + BT * 4; }
    // dS^T of one unit: 128 key rows of 64 queries (BF16), 128-byte swizzle
    static constexpr uint32_t kDSOff = kRingOff + NSB * kStageBytes;
    static constexpr uint32_t kDSBytes = FQ ? BT * BU * 2 : 0;
    static constexpr uint32_t kBarOff = kDSOff + kDSBytes;
    static constexpr int kBufs = 2;       // unit buffers in tensor memory
    // per buffer: S^T done, dP^T done (MMA commits); P^T and dS^T stored
    // (one arrival per row warp); FQ: dQ^T done (MMA commit; also frees the
    // dS^T shared-memory buffer) and dQ^T read out (one arrival per dQ warp)
    static constexpr int bKV = 0, bInFull = 1, bInEmpty = 1 + NSB, bS = 1 + 2 * NSB,
                         bDP = bS + kBufs, bDS = bDP + kBufs, bDQ = bDS + kBufs,
                         bDQFree = bDQ + kBufs, bDone = bDQFree + kBufs, kNumBars = bDone + 1;
    static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // tensor memory columns: two unit buffers {S^T, dP^T} of 64 columns each,
    // then the dV and dK accumulators. FQ packs P^T into the buffer's
    // columns 0-31 and dS^T into 32-63 (over S^T, which the row warps have
    // read), and dQ^T (M = d rows, 64 query columns) goes into 64-127 once
    // the row warps have read dP^T.
    static constexpr uint32_t cS(int b) { return 128u * b; }
    static constexpr uint32_t cDP(int b) { return 128u * b + BU; }
    static constexpr uint32_t cDV = 256, cDK = 256 + D;
    // column of K-step kk of the P^T / dS^T operand within a unit buffer
    static constexpr uint32_t p_col(int kk) { return FQ ? kk * 8 : a_col(kk); }
    static constexpr uint32_t ds_col(int kk) { return FQ ? 32 + kk * 8 : BU + a_col(kk); }
};

// --- dQ kernel: Q and dO live in tensor memory; shared memory holds a ring
// of 64-key units {K, V} ---
template <int D>
struct QCfg : BCfg<D> {
    using B = BCfg<D>;
    static constexpr int NSU = 6;                                   // unit slots
    static constexpr uint32_t kUChunkBytes = BU * B::kRowBytes;     // 64 head dims of a unit
    static constexpr uint32_t kUTileBytes = BU * D * 2;             // one 64-key K (or V) unit
    static constexpr uint32_t kRingOff = 0;
    static constexpr uint32_t k_off(int s) { return kRingOff + s * 2 * kUTileBytes; }
    static constexpr uint32_t v_off(int s) { return k_off(s) + kUTileBytes; }
    static constexpr uint32_t kBarOff = kRingOff + NSU * 2 * kUTileBytes;
    static constexpr int kBufs = 2;       // unit buffers in tensor memory
    // bQ: the row warps have stored Q and dO in tensor memory; per slot: unit
    // loaded, unit released; per buffer: S done, dP done (MMA commits), dS
    // stored (row warps)
    static constexpr int bQ = 0, bUFull = 1, bUEmpty = 1 + NSU, bS = 1 + 2 * NSU,
                         bDP = bS + kBufs, bP = bDP + kBufs, bDone = bP + kBufs,
                         kNumBars = bDone + 1;
    static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static constexpr uint32_t cS(int b) { return 128u * b; }
    static constexpr uint32_t cDP(int b) { return 128u * b + BU; }
    static constexpr uint32_t cDQ = 128u * kBufs;
    static constexpr uint32_t cQ = cDQ + D;           // Q rows, two BF16 per column
    static constexpr uint32_t cDO = cQ + D / 2;       // dO rows
    static_assert(cDO + D / 2 <= kTmemColsB, "tensor memory budget");
};

// ---------------------------------------------------------------- prep
// D = <dO_i, O_i> and LSE * log2(e) per query row. D / 8 lanes share a row,
// each reading 16 bytes of O and of dO (a warp covers 32 * 16 B of each per
// load: the kernel is a stream over O and dO), reduced by shuffles within
// the row's lanes.
template <int D>
__global__ void __launch_bounds__(256)
bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                const float* __restrict__ lse, float* __restrict__ ws_lse2,
                float* __restrict__ ws_dd, float* __restrict__ ws_dq, int Nq, int Nq_pad,
                long long rows_pad) {
    constexpr int kLanesPerRow = D / 8;
    static_assert(32 % kLanesPerRow == 0, "rows must not straddle warps");
    const long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const long long wrow = t / kLanesPerRow;
    const int sub = static_cast<int>(t % kLanesPerRow);
    const bool in = wrow < rows_pad;
    const long long bh = in ? wrow / Nq_pad : 0;
    const int i = in ? static_cast<int>(wrow % Nq_pad) : 0;
    const bool real = in && i < Nq;
    float acc = 0.f;
    if (real) {
        const long long src = (bh * Nq + i) * D + sub * 8;
        const uint4 ow = *reinterpret_cast<const uint4*>(o + src);
        const uint4 dw = *reinterpret_cast<const uint4*>(dout + src);
        const uint32_t ov[4] = {ow.x, ow.y, ow.z, ow.w}, dv[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(bf16lo_to_f32(ov[e]), bf16lo_to_f32(dv[e]), acc);
            acc = fmaf(bf16hi_to_f32(ov[e]), bf16hi_to_f32(dv[e]), acc);
        }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off >= 1; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in && ws_dq != nullptr) {
        // the dQ accumulator row starts at zero (8 values per lane)
        float4* z = reinterpret_cast<float4*>(ws_dq + wrow * D + sub * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (in && sub == 0) {
        if (real) {
            const float l = lse[bh * Nq + i];
            ws_lse2[wrow] = (l == -INFINITY) ? -INFINITY : l * kLog2eB;
            ws_dd[wrow] = acc;
        } else {
            // padding rows: lse = +inf, D = 0, so they contribute P = 0
            ws_lse2[wrow] = INFINITY;
            ws_dd[wrow] = 0.f;
        }
    }
}

// ---------------------------------------------------------------- dK, dV
// FQ: dQ is accumulated here too. After dV and dK, each unit also issues
// dQ_u^T = K^T dS_u^T (M = d, N = 64 queries, A = K read MN-major from its
// tile, B = dS_u^T from shared memory, which the row warps write beside the
// tensor-memory copy), and four dQ warps read the result out of tensor
// memory and add it into the FP32 dQ workspace with red.global.add (one
// warp instruction covers 32 consecutive head dims of one query row: 128
// contiguous bytes). The dQ accumulation order across key blocks is not
// fixed, so dQ may differ in its last bits from run to run.
template <bool FQ>
constexpr int dkdv_threads() { return (kRowWarpsB + 2 + (FQ ? 4 : 0)) * 32; }
constexpr int kDQWarp0 = kRowWarpsB + 2;

template <int D, bool FQ>
__global__ void __launch_bounds__(dkdv_threads<FQ>(), 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                const float* __restrict__ ws_lse2, const float* __restrict__ ws_dd,
                float* __restrict__ ws_dq, int H, int Nq,
                int Nk, int Nq_pad, float scale_log2, float scale, int mask_kind, int window,
                const int* __restrict__ seqlens_k, unsigned int* __restrict__ err) {
    static_assert(!FQ || (D == 128 && kRowWarpsB == 4),
                  "dQ in the keys-outer kernel: d = 128, four row warps (each owns a lane quarter)");
    using C = KVCfg<D, FQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * H + h;
    const int kb = blockIdx.x * BT;           // first key of this CTA

    int Lk = Nk;
    if (mask_kind & kMaskPadding) Lk = min(max(seqlens_k[b], 0), Nk);
    const bool causal = (mask_kind & (kMaskCausal | kMaskWindow)) != 0;
    const bool windowed = (mask_kind & kMaskWindow) != 0;
    // query blocks that see some key of [kb, min(kb + BT, Lk))
    int ilo = 0, ihi = 0;
    if (kb < Lk) {
        const int key_last = min(kb + BT, Lk) - 1;
        ilo = causal ? kb / BT : 0;
        int q_hi = Nq;                                      // exclusive
        if (windowed) q_hi = static_cast<int>(min(static_cast<long long>(Nq), static_cast<long long>(key_last) + window));
        ihi = (q_hi + BT - 1) / BT;
        if (ilo >= ihi) ilo = ihi = 0;
    }
    const int nblk = ihi - ilo;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(C::bKV), 1);
        for (int s = 0; s < NSB; ++s) {
            ptx::mbar_init(bar(C::bInFull + s), 1);
            ptx::mbar_init(bar(C::bInEmpty + s), 1);
        }
        for (int u = 0; u < C::kBufs; ++u) {
            ptx::mbar_init(bar(C::bS + u), 1);
            ptx::mbar_init(bar(C::bDP + u), 1);
            ptx::mbar_init(bar(C::bDS + u), kRowWarpsB);   // one arrival per row warp
            ptx::mbar_init(bar(C::bDQ + u), 1);
            ptx::mbar_init(bar(C::bDQFree + u), 4);          // one arrival per dQ warp
        }
        ptx::mbar_init(bar(C::bDone), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarpB) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemColsB);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProdWarp) {
        if (nblk > 0) {
            const bool leader = ptx::elect_one();
            if (leader) {
                ptx::prefetch_tmap(&tm_q);
                ptx::prefetch_tmap(&tm_do);
                ptx::mbar_arrive_expect_tx(bar(C::bKV), 2 * C::kTileBytes);
                for (int c = 0; c < D / 64; ++c) {
                    ptx::tma_load_3d(sbase + C::kKOff + c * C::kChunkBytes, &tm_k, bar(C::bKV),
                                     c * 64, kb, bh);
                    ptx::tma_load_3d(sbase + C::kVOff + c * C::kChunkBytes, &tm_v, bar(C::bKV),
                                     c * 64, kb, bh);
                }
            }
            int issued = 0;
            for (int i = 0; i < nblk; ++i) {
                const int st = i % NSB;
                const uint32_t ph = (i / NSB) & 1;
                const bool got = wait_bounded(bar(C::bInEmpty + st), ph ^ 1, abort_flag, err,
                                              kSiteKEmpty);
                if (!__all_sync(0xffffffffu, got)) break;
                if (leader) {
                    const int q0 = (ilo + i) * BT;
                    ptx::mbar_arrive_expect_tx(bar(C::bInFull + st), 2 * C::kTileBytes + C::kRowVals);
                    for (int c = 0; c < D / 64; ++c) {
                        ptx::tma_load_3d(sbase + C::q_off(st) + c * C::kChunkBytes, &tm_q,
                                         bar(C::bInFull + st), c * 64, q0, bh);
                        ptx::tma_load_3d(sbase + C::do_off(st) + c * C::kChunkBytes, &tm_do,
                                         bar(C::bInFull + st), c * 64, q0, bh);
                    }
                    const long long row = static_cast<long long>(bh) * Nq_pad + q0;
                    ptx::bulk_load(sbase + C::lse_off(st), ws_lse2 + row, BT * 4, bar(C::bInFull + st));
                    ptx::bulk_load(sbase + C::dd_off(st), ws_dd + row, BT * 4, bar(C::bInFull + st));
                }
                __syncwarp();
                issued = i + 1;
            }
            if (*abort_flag && leader) {
                wait_bounded(bar(C::bKV), 0, nullptr, err, kSiteDrain, kWaitLimitCycles / 8);
                for (int i = max(0, issued - NSB); i < issued; ++i)
                    wait_bounded(bar(C::bInFull + i % NSB), (i / NSB) & 1, nullptr, err, kSiteDrain,
                                 kWaitLimitCycles / 8);
            }
        }
    } else if (warp == kMmaWarpB) {
        if (nblk > 0) {
            const bool leader = ptx::elect_one();
            constexpr uint32_t kIdS = ptx::idesc_bf16_f32(BT, BU, false);
            constexpr uint32_t kIdG = ptx::idesc_bf16_f32(BT, D, true);
            bool ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bKV), 0, abort_flag, err, kSiteQFull));
            // Units u = 2 i + hh: query half hh of block i, tensor-memory
            // buffer u % kBufs. Issue order S(0), S(1), G(0), S(2), G(1), ...:
            // the products of unit u run while the row warps work on unit
            // u - 1, and G(u - 1) (dV, dK) follows as soon as they are done.
            static_assert(C::kBufs == 2, "G(u - 1) follows S(u); buffer = query half");
            auto do_s = [&](int i, int hh) {         // S^T, dP^T of unit 2 i + hh
                const int st = i % NSB, bf = hh, u = 2 * i + hh;
                // S^T = K Q_hh^T and dP^T = V dO_hh^T (M = 128 keys, N = 64 queries)
                const uint32_t qh = sbase + C::q_off(st) + hh * C::kUnitBytes;
                const uint32_t dh = sbase + C::do_off(st) + hh * C::kUnitBytes;
                if (leader) {
                    const uint64_t kd0 = ptx::sdesc_sw128(sbase + C::kKOff, 16, 1024);
                    const uint64_t qd0 = ptx::sdesc_sw128(qh, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
                        ptx::mma_ss(tmem + C::cS(bf), ptx::sdesc_add(kd0, off),
                                    ptx::sdesc_add(qd0, off), kIdS, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(C::bS + bf));
                }
                __syncwarp();
                if constexpr (FQ) {
                    // dP^T goes where dQ^T of unit u - 2 was: wait until the
                    // dQ warps have read it out
                    if (u >= 2) {
                        const bool got = __all_sync(
                            0xffffffffu, wait_bounded(bar(C::bDQFree + bf), ((u - 2) / 2) & 1,
                                                      abort_flag, err, kSiteODone));
                        if (!got) return false;
                        ptx::tc_fence_after();
                    }
                }
                if (leader) {
                    const uint64_t vd0 = ptx::sdesc_sw128(sbase + C::kVOff, 16, 1024);
                    const uint64_t dd0 = ptx::sdesc_sw128(dh, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
                        ptx::mma_ss(tmem + C::cDP(bf), ptx::sdesc_add(vd0, off),
                                    ptx::sdesc_add(dd0, off), kIdS, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(C::bDP + bf));
                }
                __syncwarp();
                return true;
            };
            auto do_g = [&](int i, int hh) {         // dV, dK (and dQ^T) of unit v = 2 i + hh
                const int v = 2 * i + hh, st = i % NSB, bf = hh;
                // one wait for both products: dS^T stored implies P^T stored
                const bool got = __all_sync(0xffffffffu,
                                            wait_bounded(bar(C::bDS + bf), (v / C::kBufs) & 1,
                                                         abort_flag, err, kSitePFull));
                if (!got) return false;
                ptx::tc_fence_after();
                if (leader) {
                    const uint32_t qh = sbase + C::q_off(st) + hh * C::kUnitBytes;
                    const uint32_t dh = sbase + C::do_off(st) + hh * C::kUnitBytes;
                    const uint64_t qg0 = ptx::sdesc_sw128(qh, C::kChunkBytes, 1024);
                    const uint64_t dg0 = ptx::sdesc_sw128(dh, C::kChunkBytes, 1024);
                    if constexpr (FQ) {
                        // dQ_v^T = K^T dS_v^T (M = d, N = 64 queries, K = 128 keys):
                        // A = K MN-major (head-dim atoms 16 KiB apart), B = dS^T
                        // from shared memory; 16 keys (2 KiB of rows) per step.
                        // Issued first: its completion frees the shared dS^T
                        // buffer for the next unit's row warps and starts the
                        // dQ warps' read-out.
                        constexpr uint32_t kIdQ = ptx::idesc_bf16_f32_amn(D, BU, true);
                        const uint64_t ka0 = ptx::sdesc_sw128(sbase + C::kKOff, C::kChunkBytes, 1024);
                        const uint64_t sa0 = ptx::sdesc_sw128(sbase + C::kDSOff, C::kDSBytes, 1024);
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)
                            ptx::mma_ss(tmem + C::cDP(bf), ptx::sdesc_add(ka0, kk * 16 * C::kRowBytes),
                                        ptx::sdesc_add(sa0, kk * 16 * C::kRowBytes), kIdQ,
                                        kk > 0 ? 1u : 0u);
                        ptx::mma_commit(bar(C::bDQ + bf));
                    }
                    // dV += P^T dO_hh (A from TMEM, B MN-major, K = 64 queries)
#pragma unroll
                    for (int kk = 0; kk < BU / 16; ++kk)
                        ptx::mma_ts(tmem + C::cDV, tmem + C::cS(bf) + C::p_col(kk),
                                    ptx::sdesc_add(dg0, kk * 16 * C::kRowBytes), kIdG,
                                    (v > 0 || kk > 0) ? 1u : 0u);
                    // dK += dS^T Q_hh
#pragma unroll
                    for (int kk = 0; kk < BU / 16; ++kk)
                        ptx::mma_ts(tmem + C::cDK, tmem + C::cS(bf) + C::ds_col(kk),
                                    ptx::sdesc_add(qg0, kk * 16 * C::kRowBytes), kIdG,
                                    (v > 0 || kk > 0) ? 1u : 0u);
                    // after the block's second unit, its Q/dO stage is free
                    if (hh == 1) ptx::mma_commit(bar(C::bInEmpty + st));
                }
                __syncwarp();
                return true;
            };
            auto wait_in = [&](int i) {              // Q/dO of block i landed
                const bool got = __all_sync(0xffffffffu,
                                            wait_bounded(bar(C::bInFull + i % NSB), (i / NSB) & 1,
                                                         abort_flag, err, kSiteKFull));
                if (got) ptx::tc_fence_after();
                return got;
            };
            // Block by block: S(2i), G(2i - 1), S(2i + 1), G(2i); the loop
            // body has no tests beyond the waits' own.
            if (ok && (ok = wait_in(0)) && (ok = do_s(0, 0)) && (ok = do_s(0, 1))) ok = do_g(0, 0);
            for (int i = 1; ok && i < nblk; ++i) {
                if (!(ok = wait_in(i))) break;
                if (!(ok = do_s(i, 0))) break;
                if (!(ok = do_g(i - 1, 1))) break;
                if (!(ok = do_s(i, 1))) break;
                ok = do_g(i, 0);
            }
            if (ok) ok = do_g(nblk - 1, 1);
            if (leader) ptx::mma_commit(bar(C::bDone));
            __syncwarp();
            wait_bounded(bar(C::bDone), 0, nullptr, err, kSiteDrain);
        }
    } else if (FQ && warp >= kDQWarp0) {
        // dQ warps: a warp may read only tensor-memory lane quarter warp % 4,
        // here head dims [32 qd, 32 qd + 32) of each unit's dQ^T. After the
        // read the columns are freed, and the unit's 64 query rows are added
        // into the FP32 accumulator [B*H][Nq_pad][d] with red.global.add: one
        // warp instruction covers 32 consecutive head dims of one query row,
        // a single 128-byte line. (Measured alternatives on the prefill
        // backward: 16-byte vector reductions into a head-dim-major
        // accumulator, 32 lines per instruction, 7.69 ms per step; bulk
        // tensor reductions from a shared-memory staging buffer, 7.34 ms;
        // lane pairs swapping values to issue 8-byte reductions, two lines
        // per instruction, 5.16 ms; this form 4.92-5.13 ms, against 5.52 ms
        // for recomputing S and dP in a separate dQ kernel.)
        const int qd = warp % 4;
        const int dcol = qd * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        for (int u = 0; u < 2 * nblk; ++u) {
            const int bf = u % C::kBufs;
            const bool got = wait_bounded(bar(C::bDQ + bf), (u / C::kBufs) & 1, abort_flag, err,
                                          kSiteODone);
            if (!__all_sync(0xffffffffu, got)) break;
            ptx::tc_fence_after();
            uint32_t v64[64];
            ptx::tmem_ld32x32b_x64(tmem + lane_base + C::cDP(bf), v64);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::bDQFree + bf));
            const int qb = (ilo + u / 2) * BT + (u % 2) * BU;        // first query of the unit
            float* dst = ws_dq + (static_cast<long long>(bh) * Nq_pad + qb) * D + dcol;
#pragma unroll
            for (int j = 0; j < BU; ++j) ptx::red_add_f32(dst + static_cast<long long>(j) * D,
                                                          __uint_as_float(v64[j]));
        }
    } else {
        // one thread per key row
        // warps w and w + 4 share TMEM lane quarter w % 4 (key rows); each
        // takes half of a unit's 64 query columns and, at the end, one of
        // the two accumulators (dV: warps 0-3, dK: warps 4-7)
        const int part = warp / 4;
        const int r = (warp % 4) * 32 + lane;
        const int key = kb + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
        const float2 c2 = make_float2(scale_log2, scale_log2);
        bool ok = true;
        for (int u = 0; u < 2 * nblk; ++u) {
            const int i = u / 2, hh = u % 2, bf = u % C::kBufs;
            const bool got = wait_bounded(bar(C::bS + bf), (u / C::kBufs) & 1, abort_flag, err,
                                          kSiteSFull);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            ptx::tc_fence_after();
            const int st = i % NSB;
            const int qb = (ilo + i) * BT + hh * BU;               // first query of the unit
            const float* lse2 = reinterpret_cast<const float*>(smem + C::lse_off(st)) + hh * BU;
            const float* dd = reinterpret_cast<const float*>(smem + C::dd_off(st)) + hh * BU;
            const bool full_vis = (kb + BT <= Lk) && (!causal || kb + BT - 1 <= qb) &&
                                  (!windowed || kb > qb + BU - 1 - window);
            // this key's visible queries in the unit: one interval [qb + ja, qb + je)
            int ja = 0;
            unsigned vspan = BU;
            if (!full_vis) {
                int je = BU;
                if (causal) ja = max(ja, key - qb);
                if (windowed)
                    je = static_cast<int>(min(static_cast<long long>(je),
                                              static_cast<long long>(key) + window - qb));
                if (key >= Lk) je = ja;
                vspan = static_cast<unsigned>(max(je - ja, 0));
            }
            const uint32_t a_st = tmem + lane_base + C::cS(bf);
            const uint32_t a_dpt = tmem + lane_base + C::cDP(bf);
            // Phase 1 (needs S^T): P^T = exp2(S^T c - lse2) for this warp's
            // queries (quarters of 32; LSE as 16-byte shared-memory vectors),
            // kept in FP32 for phase 2 and stored as BF16 into the first 16 of
            // the quarter's own 32 score columns (a_col), then handed to the
            // MMA warp so dV's product can start.
            float2 pf[kQuartersPerWarp][16];
#pragma unroll
            for (int k = 0; k < kQuartersPerWarp; ++k) {
                const int qt = part * kQuartersPerWarp + k;
                uint32_t sv[32];
                ptx::tmem_ld32x32b_x32(a_st + qt * 32, sv);
                float4 l4[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) l4[e] = reinterpret_cast<const float4*>(lse2)[qt * 8 + e];
                uint32_t pkp[16];
#pragma unroll
                for (int qi = 0; qi < 32; qi += 2) {
                    const float4 l = l4[qi / 4];
                    const float2 nl = (qi & 2) ? make_float2(-l.z, -l.w) : make_float2(-l.x, -l.y);
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(sv[qi]), __uint_as_float(sv[qi + 1])), c2, nl);
                    float p0 = ptx::ex2(x.x), p1 = ptx::ex2(x.y);
                    if (!full_vis) {
                        const int jq = qt * 32 + qi;
                        if (static_cast<unsigned>(jq - ja) >= vspan) p0 = 0.f;
                        if (static_cast<unsigned>(jq + 1 - ja) >= vspan) p1 = 0.f;
                    }
                    pf[k][qi / 2] = make_float2(p0, p1);
                    pkp[qi / 2] = pack_bf16x2(p0, p1);
                }
                ptx::tmem_st32x32b_x16(a_st + C::p_col(2 * qt), pkp);
            }
            // Phase 2 (needs dP^T): dS^T = P^T (dP^T - D), BF16 into the
            // quarter's own dP^T columns; one hand-off for both P^T and dS^T
            // (the wait for the stores covers every earlier one).
            const bool gotdp = wait_bounded(bar(C::bDP + bf), (u / C::kBufs) & 1, abort_flag, err,
                                            kSiteSFull);
            if (!__all_sync(0xffffffffu, gotdp)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int k = 0; k < kQuartersPerWarp; ++k) {
                const int qt = part * kQuartersPerWarp + k;
                uint32_t dpv[32];
                ptx::tmem_ld32x32b_x32(a_dpt + qt * 32, dpv);
                float4 d4[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) d4[e] = reinterpret_cast<const float4*>(dd)[qt * 8 + e];
                uint32_t pks[16];
#pragma unroll
                for (int qi = 0; qi < 32; qi += 2) {
                    const float4 dv4 = d4[qi / 4];
                    const float2 nd = (qi & 2) ? make_float2(-dv4.z, -dv4.w) : make_float2(-dv4.x, -dv4.y);
                    const float2 ds = __fmul2_rn(
                        pf[k][qi / 2],
                        __fadd2_rn(make_float2(__uint_as_float(dpv[qi]), __uint_as_float(dpv[qi + 1])),
                                   nd));
                    pks[qi / 2] = pack_bf16x2(ds.x, ds.y);
                }
                ptx::tmem_st32x32b_x16(a_st + C::ds_col(2 * qt), pks);
                if constexpr (FQ) {
                    // dS^T row r also into shared memory (B operand of dQ^T):
                    // 16-byte chunk j of the 128-byte row at j ^ (r % 8); the
                    // buffer is free once dQ^T of the previous unit is done
                    if (k == 0 && u > 0) {
                        const int pu = u - 1;
                        const bool gq = wait_bounded(bar(C::bDQ + pu % C::kBufs),
                                                     (pu / C::kBufs) & 1, abort_flag, err,
                                                     kSiteODone);
                        if (!__all_sync(0xffffffffu, gq)) { ok = false; break; }
                    }
                    const uint32_t row_addr = sbase + C::kDSOff + r * 128;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = qt * 4 + e;
                        ptx::st_shared_v4(row_addr + ((j ^ (r & 7)) << 4), pks[4 * e],
                                          pks[4 * e + 1], pks[4 * e + 2], pks[4 * e + 3]);
                    }
                }
            }
            if (!ok) break;
            if constexpr (FQ) ptx::fence_proxy_async_smem();   // dS^T stores -> tensor core
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::bDS + bf));
        }
        if (ok && nblk > 0) {
            ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bDone), 0, abort_flag, err, kSiteODone));
            ptx::tc_fence_after();
        }
        const bool have = ok && nblk > 0;
        // dV and dK leave through the V and K tiles (free once every MMA is
        // done) in the 128-byte-swizzled layout those arrived in -- 16-byte
        // piece j of key row r at j ^ (r % 8) -- and one TMA store per 64
        // head dims. (Each thread storing its own key row straight to global
        // memory touched 32 lines per warp instruction: 5.4K cycles at the
        // end of every CTA.) Rows past Nk are not stored: the copy stops at
        // the tensor's edge.
#pragma unroll
        for (int which = part; which < 2; which += kRowWarpsB / 4) {   // 0: dV, 1: dK
            const uint32_t a = tmem + lane_base + (which ? C::cDK : C::cDV);
            const float mul = which ? scale : 1.f;
            const uint32_t tile = sbase + (which ? C::kKOff : C::kVOff);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {                    // 32 head dims at a time
                uint32_t v32[32];
                if (have) {
                    ptx::tmem_ld32x32b_x32(a + cc * 32, v32);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v32[e] = 0u;
                }
                const uint32_t rbase = tile + (cc / 2) * C::kChunkBytes + r * 128;
#pragma unroll
                for (int e = 0; e < 4; ++e) {                          // 16-byte pieces
                    uint32_t pw[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f)
                        pw[f] = pack_bf16x2(__uint_as_float(v32[8 * e + 2 * f]) * mul,
                                            __uint_as_float(v32[8 * e + 2 * f + 1]) * mul);
                    const int j = (cc % 2) * 4 + e;
                    ptx::st_shared_v4(rbase + ((j ^ (r & 7)) << 4), pw[0], pw[1], pw[2], pw[3]);
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(1, 32 * kRowWarpsB);                   // every row warp
        if (warp == 0 && lane == 0) {
#pragma unroll
            for (int which = 0; which < 2; ++which)
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_store_3d(which ? &tm_dk : &tm_dv,
                                      sbase + (which ? C::kKOff : C::kVOff) + c * C::kChunkBytes,
                                      c * 64, kb, bh);
            ptx::bulk_commit_group();
            ptx::bulk_wait_read_all();            // the tiles outlive the copies' reads
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpB) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemColsB);
    }
}

// ---------------------------------------------------------------- dQ
template <int D>
__global__ void __launch_bounds__(kThreadsB, 1)
bwd_dq_kernel(const __nv_bfloat16* __restrict__ qg, const __grid_constant__ CUtensorMap tm_k64,
              const __grid_constant__ CUtensorMap tm_v64, const __nv_bfloat16* __restrict__ dog,
              const float* __restrict__ ws_lse2, const float* __restrict__ ws_dd,
              __nv_bfloat16* __restrict__ dq, int H, int Nq, int Nk, int Nq_pad, float scale_log2,
              float scale, int mask_kind, int window, const int* __restrict__ seqlens_k,
              unsigned int* __restrict__ err) {
    using C = QCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * H + h;
    const int q0 = blockIdx.x * BT;

    int Lk = Nk;
    if (mask_kind & kMaskPadding) Lk = min(max(seqlens_k[b], 0), Nk);
    const bool causal = (mask_kind & (kMaskCausal | kMaskWindow)) != 0;
    const bool windowed = (mask_kind & kMaskWindow) != 0;
    // key blocks some row of [q0, min(q0 + BT, Nq)) can see
    int jlo = 0, jhi = 0;
    {
        const int row_last = min(q0 + BT, Nq) - 1;
        int key_hi = Lk;
        if (causal) key_hi = min(key_hi, row_last + 1);
        const int key_lo = windowed ? max(0, q0 - window + 1) : 0;
        if (key_lo < key_hi) { jlo = key_lo / BT; jhi = (key_hi + BT - 1) / BT; }
    }
    const int nblk = jhi - jlo;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(C::bQ), kRowWarpsB);
        for (int s = 0; s < C::NSU; ++s) {
            ptx::mbar_init(bar(C::bUFull + s), 1);
            ptx::mbar_init(bar(C::bUEmpty + s), 1);
        }
        for (int u = 0; u < C::kBufs; ++u) {
            ptx::mbar_init(bar(C::bS + u), 1);
            ptx::mbar_init(bar(C::bDP + u), 1);
            ptx::mbar_init(bar(C::bP + u), kRowWarpsB);   // one arrival per row warp
        }
        ptx::mbar_init(bar(C::bDone), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarpB) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemColsB);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProdWarp) {
        if (nblk > 0) {
            const bool leader = ptx::elect_one();
            if (leader) {
                ptx::prefetch_tmap(&tm_k64);
                ptx::prefetch_tmap(&tm_v64);
            }
            // one 64-key unit {K, V} per slot; unit u covers keys
            // [jlo * BT + 64 u, + 64)
            int issued = 0;
            for (int u = 0; u < 2 * nblk; ++u) {
                const int st = u % C::NSU;
                const uint32_t ph = (u / C::NSU) & 1;
                const bool got = wait_bounded(bar(C::bUEmpty + st), ph ^ 1, abort_flag, err,
                                              kSiteKEmpty);
                if (!__all_sync(0xffffffffu, got)) break;
                if (leader) {
                    const int k0 = jlo * BT + u * BU;
                    ptx::mbar_arrive_expect_tx(bar(C::bUFull + st), 2 * C::kUTileBytes);
                    for (int c = 0; c < D / 64; ++c) {
                        ptx::tma_load_3d(sbase + C::k_off(st) + c * C::kUChunkBytes, &tm_k64,
                                         bar(C::bUFull + st), c * 64, k0, bh);
                        ptx::tma_load_3d(sbase + C::v_off(st) + c * C::kUChunkBytes, &tm_v64,
                                         bar(C::bUFull + st), c * 64, k0, bh);
                    }
                }
                __syncwarp();
                issued = u + 1;
            }
            if (*abort_flag && leader) {
                for (int u = max(0, issued - C::NSU); u < issued; ++u)
                    wait_bounded(bar(C::bUFull + u % C::NSU), (u / C::NSU) & 1, nullptr, err,
                                 kSiteDrain, kWaitLimitCycles / 8);
            }
        }
    } else if (warp == kMmaWarpB) {
        if (nblk > 0) {
            const bool leader = ptx::elect_one();
            constexpr uint32_t kIdS = ptx::idesc_bf16_f32(BT, BU, false);
            constexpr uint32_t kIdG = ptx::idesc_bf16_f32(BT, D, true);
            bool ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bQ), 0, abort_flag, err, kSiteQFull));
            ptx::tc_fence_after();
            // Units u: keys [jlo * BT + 64 u, + 64), ring slot u % NSU, tensor-
            // memory buffer u % kBufs. Issue order S(0), S(1), G(0), S(2),
            // G(1), ...: the products run one unit ahead of the row warps;
            // the row warps release a unit's K/V slot (below).
            const int nu = 2 * nblk;
            static_assert(C::kBufs == 2, "G(u - 1) follows S(u)");
            auto do_s = [&](int u) {                 // wait for K/V unit u; S(u), dP(u)
                const int st = u % C::NSU, bf = u % C::kBufs;
                const bool got = __all_sync(0xffffffffu,
                                            wait_bounded(bar(C::bUFull + st), (u / C::NSU) & 1,
                                                         abort_flag, err, kSiteKFull));
                if (!got) return false;
                ptx::tc_fence_after();
                if (leader) {
                    // S = Q K_u^T, dP = dO V_u^T (M = 128 queries, N = 64 keys);
                    // A = Q or dO from tensor memory (8 columns per 16 head
                    // dims), B = the K or V unit from shared memory
                    const uint64_t kd0 = ptx::sdesc_sw128(sbase + C::k_off(st), 16, 1024);
                    const uint64_t vd0 = ptx::sdesc_sw128(sbase + C::v_off(st), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t boff = (kk / 4) * C::kUChunkBytes + (kk % 4) * 32;
                        ptx::mma_ts(tmem + C::cS(bf), tmem + C::cQ + kk * 8,
                                    ptx::sdesc_add(kd0, boff), kIdS, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(C::bS + bf));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t boff = (kk / 4) * C::kUChunkBytes + (kk % 4) * 32;
                        ptx::mma_ts(tmem + C::cDP(bf), tmem + C::cDO + kk * 8,
                                    ptx::sdesc_add(vd0, boff), kIdS, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(C::bDP + bf));
                }
                __syncwarp();
                return true;
            };
            auto do_g = [&](int v) {                 // wait for dS(v); dQ += dS K_v
                const int st = v % C::NSU, bf = v % C::kBufs;
                const bool got = __all_sync(0xffffffffu,
                                            wait_bounded(bar(C::bP + bf), (v / C::kBufs) & 1,
                                                         abort_flag, err, kSitePFull));
                if (!got) return false;
                ptx::tc_fence_after();
                if (leader) {
                    // dQ += dS K_u (A = dS from TMEM, B = K MN-major, K = 64 keys)
                    const uint64_t kg0 = ptx::sdesc_sw128(sbase + C::k_off(st), C::kUChunkBytes, 1024);
#pragma unroll
                    for (int kk = 0; kk < BU / 16; ++kk)
                        ptx::mma_ts(tmem + C::cDQ, tmem + C::cS(bf) + a_col(kk),
                                    ptx::sdesc_add(kg0, kk * 16 * C::kRowBytes), kIdG,
                                    (v > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
                return true;
            };
            // S(0), then S(u), G(u - 1) for u = 1 .. nu - 1, then G(nu - 1):
            // the loop body has no tests beyond the waits' own.
            if (nu > 0) ok = ok && do_s(0);
            for (int u = 1; ok && u < nu; ++u) ok = do_s(u) && do_g(u - 1);
            if (ok && nu > 0) ok = do_g(nu - 1);
            if (leader) ptx::mma_commit(bar(C::bDone));
            __syncwarp();
            wait_bounded(bar(C::bDone), 0, nullptr, err, kSiteDrain);
        }
    } else {
        // one thread per query row
        // warps w and w + 4 share TMEM lane quarter w % 4 (query rows);
        // each takes half of a unit's 64 key columns and half of dQ's columns
        const int part = warp / 4;
        const int r = (warp % 4) * 32 + lane;
        const int row = q0 + r;
        const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
        {
            // This CTA's Q and dO rows into tensor memory (lane = row), the A
            // operands of S and dP; rows past Nq are zero. With eight row
            // warps the two warps of a lane quarter split Q and dO.
            const long long grow = (static_cast<long long>(bh) * Nq + row) * D;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                if (kRowWarpsB == 8 && which != part) continue;
                const __nv_bfloat16* src = (which ? dog : qg) + grow;
                uint32_t wv[D / 2];
#pragma unroll
                for (int e = 0; e < D / 8; ++e) {
                    uint4 u4 = make_uint4(0, 0, 0, 0);
                    if (row < Nq) u4 = reinterpret_cast<const uint4*>(src)[e];
                    wv[4 * e] = u4.x; wv[4 * e + 1] = u4.y; wv[4 * e + 2] = u4.z; wv[4 * e + 3] = u4.w;
                }
                const uint32_t dst = tmem + lane_base + (which ? C::cDO : C::cQ);
                if constexpr (D == 128) ptx::tmem_st32x32b_x64(dst, wv);
                else ptx::tmem_st32x32b_x32(dst, wv);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::bQ));
        }
        const long long wrow = static_cast<long long>(bh) * Nq_pad + row;
        const float lse2 = ws_lse2[wrow];
        const float drow = ws_dd[wrow];
        // a row that sees no key (lse = -inf) or lies past Nq (+inf) has P = 0
        const bool live = (lse2 != -INFINITY) && (lse2 != INFINITY);
        const float2 c2 = make_float2(scale_log2, scale_log2);
        // P = exp2(S c - lse2); a row that sees no key takes -inf here, so
        // every exponential is 0 without a per-element select
        const float2 nl2 = make_float2(live ? -lse2 : -INFINITY, live ? -lse2 : -INFINITY);
        const float2 nd2 = make_float2(-drow, -drow);
        bool ok = true;
        for (int u = 0; u < 2 * nblk; ++u) {
            const int j = u / 2, hh = u % 2, bf = u % C::kBufs;
            const bool got = wait_bounded(bar(C::bS + bf), (u / C::kBufs) & 1, abort_flag, err,
                                          kSiteSFull);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            // S(u) complete implies dQ(u - 2) complete (issue order S(u - 1),
            // dP(u - 1), dQ(u - 2), S(u), ...), so unit u - 2's K/V slot is
            // free: released here rather than by a commit in the MMA stream.
            if (warp == 0 && lane == 0 && u >= C::kBufs)
                ptx::mbar_arrive(bar(C::bUEmpty + (u - C::kBufs) % C::NSU));
            ptx::tc_fence_after();
            const int kb0 = (jlo + j) * BT + hh * BU;               // first key of the unit
            const bool full_vis = (kb0 + BU <= Lk) && (!causal || kb0 + BU - 1 <= q0) &&
                                  (!windowed || kb0 > q0 + BT - 1 - window);
            // this query's visible keys in the unit: one interval [kb0 + ka, kb0 + ke)
            int ka = 0;
            unsigned vspan = BU;
            if (!full_vis) {
                int ke = min(BU, Lk - kb0);
                if (causal) ke = min(ke, row + 1 - kb0);
                if (windowed) ka = max(ka, row - window + 1 - kb0);
                vspan = static_cast<unsigned>(max(ke - ka, 0));
            }
            const uint32_t a_s = tmem + lane_base + C::cS(bf);
            const uint32_t a_dp = tmem + lane_base + C::cDP(bf);
            // P for this warp's keys (quarters of 32) as soon as S is done,
            // kept in FP32 while dP's product finishes; then dS = P (dP - D)
            // in BF16 into the first 16 of the quarter's own 32 score columns.
            float2 pf[kQuartersPerWarp][16];
#pragma unroll
            for (int k = 0; k < kQuartersPerWarp; ++k) {
                const int kt = part * kQuartersPerWarp + k;
                uint32_t sv[32];
                ptx::tmem_ld32x32b_x32(a_s + kt * 32, sv);
#pragma unroll
                for (int kk = 0; kk < 32; kk += 2) {
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(sv[kk]), __uint_as_float(sv[kk + 1])), c2, nl2);
                    float p0 = ptx::ex2(x.x), p1 = ptx::ex2(x.y);
                    if (!full_vis) {
                        const int jk = kt * 32 + kk;
                        if (static_cast<unsigned>(jk - ka) >= vspan) p0 = 0.f;
                        if (static_cast<unsigned>(jk + 1 - ka) >= vspan) p1 = 0.f;
                    }
                    pf[k][kk / 2] = make_float2(p0, p1);
                }
            }
            const bool gotdp = wait_bounded(bar(C::bDP + bf), (u / C::kBufs) & 1, abort_flag, err,
                                            kSiteSFull);
            if (!__all_sync(0xffffffffu, gotdp)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int k = 0; k < kQuartersPerWarp; ++k) {
                const int kt = part * kQuartersPerWarp + k;
                uint32_t dpv[32];
                ptx::tmem_ld32x32b_x32(a_dp + kt * 32, dpv);
                uint32_t pks[16];
#pragma unroll
                for (int kk = 0; kk < 32; kk += 2) {
                    const float2 ds = __fmul2_rn(
                        pf[k][kk / 2],
                        __fadd2_rn(make_float2(__uint_as_float(dpv[kk]), __uint_as_float(dpv[kk + 1])),
                                   nd2));
                    pks[kk / 2] = pack_bf16x2(ds.x, ds.y);
                }
                ptx::tmem_st32x32b_x16(a_s + kt * 32, pks);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::bP + bf));
        }
        if (ok && nblk > 0) {
            ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bDone), 0, abort_flag, err, kSiteODone));
            ptx::tc_fence_after();
        }
        const bool have = ok && nblk > 0;
        __nv_bfloat16* dst = dq + (static_cast<long long>(bh) * Nq + row) * D;
        constexpr int kChunksPerWarp = (D / 32) / (kRowWarpsB / 4);
#pragma unroll
        for (int cc = part * kChunksPerWarp; cc < (part + 1) * kChunksPerWarp; ++cc) {
            uint32_t v32[32];
            if (have) {
                ptx::tmem_ld32x32b_x32(tmem + lane_base + C::cDQ + cc * 32, v32);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v32[e] = 0u;
            }
            if (row < Nq) {
                uint32_t pw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pw[e] = pack_bf16x2(__uint_as_float(v32[2 * e]) * scale,
                                        __uint_as_float(v32[2 * e + 1]) * scale);
                uint4* o4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o4[e] = make_uint4(pw[4 * e], pw[4 * e + 1], pw[4 * e + 2], pw[4 * e + 3]);
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpB) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemColsB);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes, int* configured) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (*configured == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) *configured = dev;
    return e;
}

// dQ = scale * (FP32 accumulator [B*H][Nq_pad][d]) rounded to BF16 for the
// real query rows; eight head dims per thread (two 16-byte loads, one
// 16-byte store).
template <int D>
__global__ void __launch_bounds__(256)
bwd_dq_convert_kernel(const float* __restrict__ ws_dq, __nv_bfloat16* __restrict__ dq,
                      long long rows, int Nq, int Nq_pad, float scale) {
    constexpr int kPer = D / 8;
    const long long n = rows * kPer;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = t / kPer;            // (bh, q) over the real rows
        const int part = static_cast<int>(t % kPer);
        const long long bh = row / Nq;
        const long long q = row - bh * Nq;
        const float4* src = reinterpret_cast<const float4*>(ws_dq + (bh * Nq_pad + q) * D + part * 8);
        const float4 a = src[0], b = src[1];
        uint4 w;
        w.x = pack_bf16x2(a.x * scale, a.y * scale);
        w.y = pack_bf16x2(a.z * scale, a.w * scale);
        w.z = pack_bf16x2(b.x * scale, b.y * scale);
        w.w = pack_bf16x2(b.z * scale, b.w * scale);
        *reinterpret_cast<uint4*>(dq + row * D + part * 8) = w;
    }
}

#ifndef ATTN_BWD_FUSED_DQ
#define ATTN_BWD_FUSED_DQ 1
#endif

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                         const CUtensorMap& tdv, const CUtensorMap& tk64, const CUtensorMap& tv64,
                         cudaStream_t stream) {
    constexpr bool FQ = (D == 128) && ATTN_BWD_FUSED_DQ != 0;
    static int cfg_kv = -1, cfg_q = -1;
    cudaError_t e = set_smem(bwd_dkdv_kernel<D, FQ>, KVCfg<D, FQ>::kSmemBytes, &cfg_kv);
    if (e != cudaSuccess) return e;
    if (!FQ) {
        e = set_smem(bwd_dq_kernel<D>, QCfg<D>::kSmemBytes, &cfg_q);
        if (e != cudaSuccess) return e;
    }
    const int Nq_pad = (a.Nq + BT - 1) / BT * BT;
    const long long rows_pad = static_cast<long long>(a.B) * a.H * Nq_pad;
    const float scale_log2 = a.scale * kLog2eB;
    const long long prep_threads = rows_pad * (D / 8);
    float* ws_dq = FQ ? a.ws_dq : nullptr;
    bwd_prep_kernel<D><<<static_cast<unsigned>((prep_threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
        a.ws_lse2, a.ws_dd, ws_dq, a.Nq, Nq_pad, rows_pad);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    dim3 g1((a.Nk + BT - 1) / BT, a.H, a.B);
    bwd_dkdv_kernel<D, FQ><<<g1, dkdv_threads<FQ>(), KVCfg<D, FQ>::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, tdk, tdv, a.ws_lse2, a.ws_dd, ws_dq, a.H, a.Nq, a.Nk, Nq_pad, scale_log2,
        a.scale,
        a.mask_kind, a.window, a.seqlens_k, a.err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (FQ) {
        const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
        const long long threads = rows * (D / 8);
        const unsigned blocks =
            static_cast<unsigned>(std::min<long long>((threads + 255) / 256, 152LL * 16));
        bwd_dq_convert_kernel<D><<<blocks, 256, 0, stream>>>(
            ws_dq, static_cast<__nv_bfloat16*>(a.dq), rows, a.Nq, Nq_pad, a.scale);
        return cudaGetLastError();
    }
    dim3 g2((a.Nq + BT - 1) / BT, a.H, a.B);
    bwd_dq_kernel<D><<<g2, kThreadsB, QCfg<D>::kSmemBytes, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), tk64, tv64,
        static_cast<const __nv_bfloat16*>(a.dout), a.ws_lse2, a.ws_dd, static_cast<__nv_bfloat16*>(a.dq), a.H, a.Nq, a.Nk,
        Nq_pad, scale_log2, a.scale, a.mask_kind, a.window, a.seqlens_k, a.err);
    return cudaGetLastError();
}

}  // namespace

bool bwd_fused_dq(int d) { return d == 128 && ATTN_BWD_FUSED_DQ != 0; }

cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const CUtensorMap& tk64, const CUtensorMap& tv64,
                       cudaStream_t stream) {
    return a.d == 64 ? launch_bwd_d<64>(a, tq, tk, tv, tdo, tdk, tdv, tk64, tv64, stream)
                     : launch_bwd_d<128>(a, tq, tk, tv, tdo, tdk, tdv, tk64, tv64, stream);
}

}  // namespace attn
