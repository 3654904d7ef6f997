// fwd_sm103.cu -- fused attention forward (BF16 or E4M3 inputs) on the sm_103a tensor cores.
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
// "Common mistakes", on causal masking).
//
// Rescaling. P2 ("What interviewers probe next") notes that alpha is exactly 1
// when the max does not change, and that the FlashAttention-4 variant goes
// further: it moves the reference only when the max grows past a threshold,
// which stays exact because l and A share the reference and the final
// division cancels it. This kernel does the latter: each row keeps a
// reference m_use that moves to the block max only when that exceeds m_use by
// more than kTau = 8 (log2 units), so P <= 2^8, and A is rescaled in tensor
// memory only for warps where some row moved; lse = m_use + log l.
//
// GB300 mapping (one CTA per SM, 352 threads):
//   * Two query tiles per CTA (256 rows) share every K/V block, so each
//     block is read from device memory once per 256 queries, and the tensor
//     core works on one tile's products while the other tile's softmax runs.
//   * Warp 8 issues TMA bulk-tensor loads of each tile's Q (once, on a
//     barrier per tile) and of the first K block before the CTA's set-up,
//     which they overlap -- tile 0's first S product waits for its own Q
//     and K only -- and streams K_j into a 3-slot ring; warp 10 streams V_j
//     into a 2-slot ring (5 and 4 at d = 64, 6 and 5 for E4M3);
//     128-byte-swizzled shared-memory buffers.
//     K_j and V_{j-1}, the inputs of one MMA step, complete on one mbarrier
//     with transaction counts, so the MMA warp waits once per step (each
//     wait in its issue stream costs the tensor pipe: one wait fewer per
//     block measured 1.415 -> 1.346 ms on the prefill).
//   * Operand descriptors are built once per MMA group and advanced by the
//     byte offset of each K-step (the issuing lane is on the critical path:
//     this alone was worth 4 % of throughput).
//   * Warp 9 allocates 512 tensor-memory columns (S_0, S_1, O_0, O_1; FP32)
//     and runs the MMA schedule as a whole warp (uniform control flow, so the
//     loop state and operand descriptors stay in uniform registers); one
//     lane elected with elect.sync issues every tcgen05.mma: S_t = Q_t K_j^T with both
//     operands in shared memory, and O_t += P_t V_j with P_t read from tensor
//     memory (BF16, written over S_t) and V_j from shared memory. Issue order
//     per block: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j). The MMA warp commits
//     only S and the final O; the K and V slots are released by the softmax
//     warp that sees the block's last S product complete. CTAs whose tiles
//     cover the same blocks (and causal ones, whose key blocks are walked
//     from the diagonal down so that tile 0 starts one step after tile 1)
//     run a straight-line version of the schedule without per-tile range
//     tests.
//   * Warps 0-3 run the softmax of tile 0 and warps 4-7 that of tile 1, one
//     thread per query row: tcgen05.ld of the 128 scores of its row, mask,
//     row max (four independent three-input max chains) and row sum (packed
//     FP32x2 adds) in registers -- no shuffles, the row is in one thread --,
//     exp2 with the scale folded into one packed FMA, P stored back to tensor
//     memory in two 64-key halves and signalled once, after both (the MMA
//     warp reaches a tile's P V product well after its P is ready, so a
//     separate hand-off per half only adds a wait to the issue stream: one
//     hand-off per tile measured 1.507 -> 1.439 ms on the prefill); then
//     the epilogue O = A / l and lse, O leaving through the tile's dead Q
//     buffer, one TMA store per 64 head dims as soon as it is staged (E4M3:
//     in two passes through the half-size buffer).
//   * m, l and A are FP32; P is rounded to BF16 for the P V product.
//   * Exponentials: ex2.approx on the MUFU unit; a compile-time fraction of
//     them runs as a polynomial on the FMA pipe instead (soft_exp2x2:
//     relative error 1.02e-4, below P's BF16 rounding): none for BF16, 1 of
//     every 16 pairs for E4M3 by default.
//   * E4M3 variant (d = 128): Q, K and V are 8-bit floats with per-tensor
//     dequantisation factors, the FP8 mode that P1 ("What did
//     FlashAttention-2 and -3 change?") and P3 ("Where the merge is used
//     today") credit to FlashAttention-3. Both products run as
//     kind::f8f6f4 (K = 32 per instruction, half the MMA issue of BF16), P
//     is rounded to E4M3 (P <= 2^8 < 448, the format's largest finite value)
//     and stored four per tensor-memory column, the Q and K factors fold
//     into the exp2 scale and V's into the final 1/l; m, l, A stay FP32 and
//     O is BF16. Tiles are half the bytes, so the K and V rings are deeper.
//   * Every mbarrier wait is bounded; on expiry the CTA records the site in
//     the device error word, all roles stop, in-flight copies and MMAs are
//     drained, tensor memory is freed and the kernel returns.
//   * CTA-pair form (PAIR, BF16 at d = 128; a compile-time choice of the
//     library, off by default). Clusters of two CTAs own four tiles; tile t
//     of the pair is one M = 256 MMA (tcgen05 cta_group::2) over 128 rows of
//     each CTA. Each CTA loads half of every K block (64 keys) and half of
//     every V block (64 head dims), so the tensor cores read half as much B
//     operand from each SM's shared memory. The first CTA issues every MMA;
//     its commits arrive on both CTAs' barriers (multicast), both CTAs'
//     copies count on its step barriers (cta_group::2 TMA), and the second
//     CTA's softmax warps hand P over by remote arrivals on its P barriers.
//     Same arithmetic as the one-CTA kernel (identical results in key
//     order; under causal masks the one-CTA kernel walks the blocks from the
//     diagonal down, and the two agree to rounding), but slower
//     on GB300 (prefill B1 H64 8192^2: 1.49-1.65 against 1.29-1.34 ms; tensor
//     pipe 57 % against 74 % active): the forward's pace is set by the
//     softmax -> P -> MMA hand-off, and in a pair every hand-off crosses to
//     the other SM and waits for the slower of two softmaxes.
#include <algorithm>
#include <climits>
#include "common.cuh"

namespace attn {
namespace {

constexpr int BM = 128;                 // query rows per tile
constexpr int NT = 2;                   // query tiles per CTA
constexpr int BN = 128;                 // keys per block
constexpr int kSoftmaxWarps = 4 * NT;
constexpr int kProducerWarp = kSoftmaxWarps;       // Q and K loads
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kProducerVWarp = kSoftmaxWarps + 2;  // V loads
constexpr int kThreads = (kSoftmaxWarps + 3) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy-rescale threshold in log2 units: the row's reference max moves only
// when a block's max exceeds it by more than this (P stays <= 2^kTau = 256).
constexpr float kTau = 8.0f;
// Of every 16 pairs of exponentials of P, this many are computed in software
// on the FMA pipe (soft_exp2x2) and the rest by ex2.approx on the MUFU unit,
// spread evenly through the group (a compile-time choice). With the MMA
// issue stream slimmed down the softmax has slack and every extra
// instruction in it shows: prefill B1 H64 8192^2 d128 1.312 / 1.319 /
// 1.378 ms with 0 / 1 / 2 pairs (BF16), causal 0.731 / 0.744 / 0.763 ms,
// E4M3 1.064 / 1.110 ms with 0 / 1. (An earlier build, whose softmax was
// on the critical path, measured 1 pair fastest for BF16.) Since the E4M3
// kernel runs the straight-line schedule, its exponential unit is the
// tighter resource there: E4M3 prefill 1.072 / 1.067 / 1.084 ms with
// 0 / 1 / 2 pairs, BF16 still slower with 1. The polynomial's relative error
// (1.0e-4) is far below P's rounding to E4M3 (2^-4).
#ifndef ATTN_SOFT_EXP2_PAIRS_BF16
#define ATTN_SOFT_EXP2_PAIRS_BF16 0
#endif
#ifndef ATTN_SOFT_EXP2_PAIRS_E4M3
#define ATTN_SOFT_EXP2_PAIRS_E4M3 1
#endif
template <bool F8>
__host__ __device__ constexpr bool soft_pair(int idx) {
    constexpr int k = F8 ? ATTN_SOFT_EXP2_PAIRS_E4M3 : ATTN_SOFT_EXP2_PAIRS_BF16;
    static_assert(k >= 0 && k <= 16, "pairs per group of 16");
    return (idx * k) % 16 < k;
}

// F8 = false: BF16 Q, K, V (kind::f16, K = 16 per MMA); F8 = true: E4M3
// Q, K, V (kind::f8f6f4, K = 32 per MMA), d = 128 only. PAIR: the CTA-pair
// form (BF16, d = 128): each MMA spans the tensor cores of two SMs (M = 256,
// 128 query rows from each CTA) and each CTA holds half of every K block
// (64 keys) and half of every V block (64 head dims).
template <int D, bool F8, bool PAIR = false>
struct Cfg {
    static_assert(!PAIR || (D == 128 && !F8), "the CTA-pair form is BF16 with d = 128");
    static constexpr int kElem = F8 ? 1 : 2;                   // bytes per element
    static_assert((D * kElem) % 128 == 0, "head dim must fill 128-byte swizzle rows");
    // K/V ring depths: K is consumed one MMA step ahead of V, so it gets the
    // deeper ring (BF16, d = 128: Q 64 KiB + K 3 x 32 KiB + V 2 x 32 KiB =
    // 224 KiB; E4M3: Q 32 KiB + K 6 x 16 KiB + V 5 x 16 KiB = 208 KiB, 1 %
    // faster than 4 + 4 on the E4M3 prefill; pair: Q 64 KiB + K 5 x 16 KiB +
    // V 4 x 16 KiB = 208 KiB). The V ring must be the shallower one: step
    // barriers (one per K slot) also carry V.
    static constexpr int kStagesK = PAIR ? 5 : F8 ? 6 : (D == 64) ? 5 : 3;
    static constexpr int kStagesV = PAIR ? 4 : F8 ? 5 : (D == 64) ? 4 : 2;
    static_assert(kStagesV < kStagesK, "a V load may not reach a step barrier's next phase");
    static constexpr int kCtas = PAIR ? 2 : 1;                 // CTAs sharing one MMA
    static constexpr int kMmaM = BM * kCtas;                   // query rows per MMA
    static constexpr uint32_t kRowBytes = 128;                 // one swizzle atom row
    static constexpr int kChunkElems = 128 / kElem;            // head dims per atom row
    static constexpr int kChunks = D * kElem / 128;
    static constexpr int kQKSteps = D * kElem / 32;            // MMAs of S = Q K^T (32 B of K each)
    static constexpr int kPVKeys = 32 / kElem;                 // keys per P V MMA
    static constexpr int kPVSteps = BN / kPVKeys;               // P V MMAs per block
    static constexpr uint32_t kPHalfCols = (BN / 2) * kElem / 4;   // TMEM columns of half of P
    static constexpr uint32_t kQTileBytes = BM * D * kElem;
    static constexpr uint32_t kKVBytes = BN * D * kElem;       // a whole K or V block
    static constexpr uint32_t kSlotBytes = kKVBytes / kCtas;   // this CTA's share of one
    static constexpr int kKRows = BN / kCtas;                  // keys of a K block held here
    static constexpr uint32_t kQChunkBytes = BM * kRowBytes;   // one atom column of a Q tile
    static constexpr uint32_t kKChunkBytes = kKRows * kRowBytes;   // one atom column of a K slot
    static constexpr uint32_t kVChunkBytes = BN * kRowBytes;   // one atom column of a V slot
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKOff = kQOff + NT * kQTileBytes;
    static constexpr uint32_t kVOff = kKOff + kStagesK * kSlotBytes;
    static constexpr uint32_t kBarOff = kVOff + kStagesV * kSlotBytes;
    // barrier indices (pair: QFull, Step and PFull are used in the first
    // CTA only, where the MMAs are issued; the others in both)
    static constexpr int bQFull = 0;                   // [NT]: tile t's Q landed
    static constexpr int bStep = bQFull + NT;          // [NSK]: step s has K_s and V_{s-1}
    static constexpr int bKEmpty = bStep + kStagesK;
    static constexpr int bVEmpty = bKEmpty + kStagesK;
    static constexpr int bSFull = bVEmpty + kStagesV;
    static constexpr int bPFull = bSFull + NT;         // [NT]: P of the tile's block stored
    static constexpr int bODone = bPFull + NT;
    static constexpr int bDrain = bODone + NT;
    static constexpr int kNumBars = bDrain + 1;
    static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag
    static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static constexpr uint32_t s_col(int t) { return t * BN; }
    static constexpr uint32_t o_col(int t) { return NT * BN + t * D; }
    static_assert(NT * BN + NT * D <= kTmemCols, "tensor memory budget");
};

struct Range { int lo, hi; };   // key blocks [lo, hi)

// Key blocks that some row of [row_first, row_first + rows) can see.
__device__ __forceinline__ Range tile_range(int row_first, int rows, int Nq, int Lk, bool causal,
                                            bool windowed, int window) {
    if (row_first >= Nq) return {0, 0};
    const int row_last = min(row_first + rows, Nq) - 1;
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

// 352 threads, one CTA per SM. The register file is split by sub-partition
// (16,384 each) and three of the eleven warps share one, so a thread gets at
// most 168 registers. PAIR: launched in clusters of two CTAs (x), which
// together own four query tiles; CTA 0 issues every MMA of the pair.
template <int D, bool F8, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
fwd_sm103_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 __nv_bfloat16* __restrict__ o_ptr, float* __restrict__ lse, int H, int Nq, int Nk,
                 float scale_log2, float o_mul, int mask_kind, int window,
                 const int* __restrict__ seqlens_k, unsigned int* __restrict__ err,
                 int group_heads) {
    using C = Cfg<D, F8, PAIR>;
    constexpr int NSK = C::kStagesK, NSV = C::kStagesV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // rank in the pair (0 issues the MMAs); the pair's barriers that collect
    // both CTAs' copies and P hand-offs live in CTA 0, addressed through
    // the cluster window.
    const int rank = PAIR ? static_cast<int>(ptx::cluster_ctarank()) : 0;
    const bool issuer_cta = rank == 0;
    auto lead_bar = [&](int i) -> uint32_t {
        if constexpr (PAIR) return ptx::mapa_shared(bar(i), 0);
        else return bar(i);
    };
    // Unmasked (group_heads == 0): the units of one head are adjacent (they
    // share K and V in L2). Causal or windowed: the heads are taken in groups
    // of group_heads, and within a group the longest units of every head
    // come first, so the last wave holds the shortest CTAs instead of one
    // head's longest ones, while the K and V of the heads in flight (one
    // group, two at a group boundary) stay within L2 (all heads at once
    // re-read K and V from device memory about five times on the causal
    // workload). A unit is the NT tiles of one CTA, or of a CTA pair.
    const int units = gridDim.x / C::kCtas;
    int unit = blockIdx.x / C::kCtas, h = blockIdx.y, b = blockIdx.z;
    if (group_heads > 0) {
        // 32-bit arithmetic (the launcher keeps the grid below 2^31 CTAs; a
        // 64-bit division is a long software sequence on the CTA's start-up
        // path)
        const int nbh = gridDim.y * gridDim.z;
        const int lin = unit + units * (blockIdx.y + gridDim.y * blockIdx.z);
        const int per_group = group_heads * units;
        const int g = lin / per_group;
        const int idx = lin - g * per_group;
        const int gh = min(group_heads, nbh - g * group_heads);   // heads in this group
        unit = units - 1 - idx / gh;
        const int bhl = g * group_heads + idx % gh;
        h = bhl % H;
        b = bhl / H;
    }
    const int bh = b * H + h;
    // Tile t of the unit covers rows [q0 + t * kMmaM, + kMmaM); this CTA's
    // share of it starts at own_row(t).
    const int q0 = unit * (C::kMmaM * NT);
    auto own_row = [&](int t) { return q0 + t * C::kMmaM + rank * BM; };

    int Lk = Nk;
    if (mask_kind & kMaskPadding) Lk = min(max(seqlens_k[b], 0), Nk);
    const bool causal = (mask_kind & (kMaskCausal | kMaskWindow)) != 0;
    const bool windowed = (mask_kind & kMaskWindow) != 0;

    // Key-block ranges of the MMA tiles (pair: the union over both CTAs'
    // rows, identical in both CTAs)
    Range R[NT];
    int lo = INT_MAX, hi = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        R[t] = tile_range(q0 + t * C::kMmaM, C::kMmaM, Nq, Lk, causal, windowed, window);
        if (R[t].lo < R[t].hi) { lo = min(lo, R[t].lo); hi = max(hi, R[t].hi); }
    }
    if (hi == 0) {
        // No row of this CTA (or pair) sees a key: O = 0 and lse = -inf for
        // its rows, written directly -- no barriers, tensor memory or loads.
        // (Under padding and sliding windows a large share of CTAs are empty.)
        __nv_bfloat16* ob = o_ptr + static_cast<long long>(bh) * Nq * D;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int r0 = own_row(t);
            const int rows = max(0, min(BM, Nq - r0));
            uint4* dst = reinterpret_cast<uint4*>(ob + static_cast<long long>(r0) * D);
            for (int e = threadIdx.x; e < rows * D / 8; e += kThreads) dst[e] = make_uint4(0u, 0u, 0u, 0u);
            if (lse != nullptr)
                for (int e = threadIdx.x; e < rows; e += kThreads)
                    lse[static_cast<long long>(bh) * Nq + r0 + e] = -INFINITY;
        }
        return;
    }
    // Under a causal mask tile 1 sees one key block more than tile 0: the
    // diagonal block of its own rows, the last in key order. Walked in key
    // order it would run alone at the end (tile 1's S -> softmax -> P V chain
    // with nothing to overlap it); so such CTAs walk their key blocks from
    // the last down, and the extra block becomes the first step, where tile 0
    // is still waiting for its Q anyway. The schedule below works on steps:
    // the ranges R[t] become step ranges (offset by lo), and blk() maps a
    // step's block back to the key block that is loaded and masked.
    const bool rev = !PAIR && causal && R[0].lo == lo && R[1].lo == lo && R[1].hi == hi &&
                     R[0].hi == hi - 1;
    if (rev) R[0] = Range{lo + 1, hi};
    auto blk = [&](int v) { return rev ? lo + hi - 1 - v : v; };
    // Tile 1 starting inside tile 0's range, one block later (a sliding
    // window; the straight-line schedule's late1 case below): its first S
    // product is issued at the start of that step, ahead of tile 0's P V
    // product of the previous block, so that its softmax does not wait for
    // tile 0's first one. That step's K and V blocks are then last read by
    // tile 0's S product, and tile 0's softmax releases them (see the
    // release rule below).
    const int early_s = (!PAIR && R[1].lo > R[0].lo && R[1].lo < R[0].hi && R[1].lo < R[1].hi)
                            ? R[1].lo : -1;
    // This CTA's Q tiles, loaded into its own shared memory; completion is
    // counted on the issuing CTA's barrier. Only tiles that see some key: an
    // empty tile's buffer is written by its epilogue straight away and must
    // not receive a late Q.
    auto load_q = [&](int t) {
        if (R[t].lo >= R[t].hi) return;
        for (int c = 0; c < C::kChunks; ++c) {
            const uint32_t dst = sbase + C::kQOff + t * C::kQTileBytes + c * C::kQChunkBytes;
            if constexpr (PAIR)
                ptx::tma_load_3d_pair(dst, &tm_q, lead_bar(C::bQFull + t), c * C::kChunkElems,
                                      own_row(t), bh);
            else
                ptx::tma_load_3d(dst, &tm_q, bar(C::bQFull + t), c * C::kChunkElems, own_row(t), bh);
        }
    };

    // The Q tiles and the first K block are the first things the CTA needs
    // and the longest loads it waits for: the thread that sets up the
    // barriers starts them before the tensor-memory allocation and the
    // block-wide barrier (pair: the second CTA's Q, which counts on the
    // first CTA's barrier, after the cluster barrier that publishes its
    // initialisation; the pair's K blocks all come from the producer loop).
    // One CTA: K_lo goes into slot 0 of the K ring on step barrier 0, as the
    // producer loop would load it (a fresh ring has every slot free), right
    // after tile 0's Q: with one Q barrier per tile, tile 0's first S product
    // waits for 64 KiB (BF16) instead of both Q tiles and K_lo.
    if (warp == kProducerWarp && lane == 0) {
        for (int t = 0; t < NT; ++t) ptx::mbar_init(bar(C::bQFull + t), 1);
        for (int s = 0; s < NSK; ++s) {
            ptx::mbar_init(bar(C::bStep + s), 2);            // the K and the V producer
            ptx::mbar_init(bar(C::bKEmpty + s), 1);
        }
        for (int s = 0; s < NSV; ++s) ptx::mbar_init(bar(C::bVEmpty + s), 1);
        for (int t = 0; t < NT; ++t) {
            ptx::mbar_init(bar(C::bSFull + t), 1);
            ptx::mbar_init(bar(C::bPFull + t), 4 * C::kCtas);   // one arrival per softmax warp
            ptx::mbar_init(bar(C::bODone + t), 1);
        }
        ptx::mbar_init(bar(C::bDrain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        if (lo < hi && issuer_cta) {
            ptx::prefetch_tmap(&tm_q);
            auto start_q = [&](int t) {
                if (R[t].lo < R[t].hi) {
                    ptx::mbar_arrive_expect_tx(bar(C::bQFull + t), C::kCtas * C::kQTileBytes);
                    load_q(t);
                }
            };
            // the Q of the tile whose first S comes first, the first K block,
            // then the other Q
            if (rev) start_q(1); else start_q(0);
            if constexpr (!PAIR) {
                ptx::prefetch_tmap(&tm_k);
                ptx::mbar_arrive_expect_tx(bar(C::bStep), C::kKVBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    ptx::tma_load_3d(sbase + C::kKOff + c * C::kKChunkBytes, &tm_k, bar(C::bStep),
                                     c * C::kChunkElems, blk(lo) * BN, bh);
            }
            if (rev) start_q(0); else start_q(1);
        }
        // the O map, used by the epilogue's stores (one-CTA BF16 form; E4M3
        // measured 1 % slower with it, and the pair form spills registers)
        if constexpr (!F8 && !PAIR) ptx::prefetch_tmap(&tm_o);
    }
    if (warp == kMmaWarp) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    if constexpr (PAIR) {
        ptx::cluster_arrive_release();
        ptx::cluster_wait_acquire();
        if (warp == kProducerWarp && lane == 0 && lo < hi && !issuer_cta) {
            ptx::prefetch_tmap(&tm_q);
            for (int t = 0; t < NT; ++t) load_q(t);
        }
    } else {
        __syncthreads();
    }
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp || warp == kProducerVWarp) {
        // ------------------------------------------------------ TMA producers
        // Warp 8 (which started the Q loads above) streams K; warp 10
        // streams V. Each ring is refilled as soon as a slot is released (by
        // the softmax warp that sees the block's last S product complete).
        // Step i = s - lo of the MMA schedule reads K_s and V_{s-1}; both
        // loads complete on step barrier i % NSK, which takes one arrival
        // from each producer per phase (a plain one where the step has no
        // such block: no V at the first step, no K at the last), so the MMA
        // warp waits once per step. A producer arrives on step i's barrier
        // only after the release of a block consumed at step i - NSK or
        // later (K: K_{i-NSK}; V: V_{i-1-NSV}, with NSV < NSK), so the
        // barrier's previous phase is always complete. The whole warp runs
        // the loop (uniform control flow); one elected lane issues.
        if (lo < hi) {
            const bool leader = ptx::elect_one();
            const bool is_k = (warp == kProducerWarp);
            const int ns = is_k ? NSK : NSV;
            const int empty0 = is_k ? C::bKEmpty : C::bVEmpty;
            const uint32_t ring = sbase + (is_k ? C::kKOff : C::kVOff);
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            if (leader) ptx::prefetch_tmap(map);
            const int n = hi - lo;
            int issued = 0;                          // blocks whose copy has started
            for (int i = 0; i <= n; ++i) {
                const int b = is_k ? i : i - 1;      // block this producer adds to step i
                const bool load = b >= 0 && b < n;
                const uint32_t sb = bar(C::bStep + i % NSK);
                if (!PAIR && is_k && b == 0) {
                    issued = 1;                      // started with the Q tiles
                } else if (load) {
                    const int st = b % ns;
                    const bool got = wait_bounded(bar(empty0 + st), ((b / ns) & 1) ^ 1, abort_flag,
                                                  err, is_k ? kSiteKEmpty : kSiteVEmpty);
                    if (!__all_sync(0xffffffffu, got)) break;
                    if (leader) {
                        // The issuing CTA's producer expects the whole block
                        // (pair: both CTAs' halves, which count on its barrier).
                        if (issuer_cta) ptx::mbar_arrive_expect_tx(sb, C::kKVBytes);
                        const uint32_t dst = ring + st * C::kSlotBytes;
                        if constexpr (PAIR) {
                            // K: keys [64 rank, + 64) of the block, every head
                            // dim; V: every key, head dims [64 rank, + 64).
                            const uint32_t lsb = lead_bar(C::bStep + i % NSK);
                            if (is_k) {
                                for (int c = 0; c < C::kChunks; ++c)
                                    ptx::tma_load_3d_pair(dst + c * C::kKChunkBytes, map, lsb,
                                                          c * C::kChunkElems,
                                                          blk(lo + b) * BN + rank * C::kKRows, bh);
                            } else {
                                ptx::tma_load_3d_pair(dst, map, lsb, rank * C::kChunkElems,
                                                      blk(lo + b) * BN, bh);
                            }
                        } else {
                            const uint32_t chunk = is_k ? C::kKChunkBytes : C::kVChunkBytes;
                            for (int c = 0; c < C::kChunks; ++c)
                                ptx::tma_load_3d(dst + c * chunk, map, sb, c * C::kChunkElems,
                                                 blk(lo + b) * BN, bh);
                        }
                    }
                    issued = b + 1;
                } else if (issuer_cta) {
                    // no block for this step: K at the last step; V at the
                    // first. K's last-step arrival waits like a load would,
                    // for the release of K_{n-NSK}.
                    if (is_k && n >= NSK) {
                        const bool got = wait_bounded(bar(empty0 + n % NSK), ((n / NSK) & 1) ^ 1,
                                                      abort_flag, err, kSiteKEmpty);
                        if (!__all_sync(0xffffffffu, got)) break;
                    }
                    if (leader) ptx::mbar_arrive(sb);
                }
                __syncwarp();
            }
            if (*abort_flag && leader) {
                // Let the copies this warp started land before the CTA exits
                // (bounded: a step's phase also needs the other producer).
                if (issuer_cta) {
                    if (is_k)
                        for (int t = 0; t < NT; ++t)
                            if (R[t].lo < R[t].hi)
                                wait_bounded<PAIR>(bar(C::bQFull + t), 0, nullptr, err, kSiteDrain,
                                                   kWaitLimitCycles / 8);
                    for (int b = max(0, issued - ns); b < issued; ++b) {
                        const int i = is_k ? b : b + 1;
                        wait_bounded<PAIR>(bar(C::bStep + i % NSK), (i / NSK) & 1, nullptr, err,
                                           kSiteDrain, kWaitLimitCycles / 8);
                    }
                } else {
                    // pair, second CTA: its copies count on the first CTA's
                    // barriers, which it cannot wait on; give them time to land
                    const long long t0 = clock64();
                    while (clock64() - t0 < 200000) { }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        // The whole warp runs the schedule and waits; one elected lane issues
        // every tcgen05.mma / tcgen05.commit, so the loop state and the
        // operand descriptors stay warp-uniform. Pair: only the first CTA
        // issues; its commits arrive on the barrier at the same offset in
        // both CTAs.
        if (lo < hi && issuer_cta) {
            const bool leader = ptx::elect_one();
            constexpr uint32_t kIdescS = F8 ? ptx::idesc_e4m3_f32(BM, BN, false)
                                            : ptx::idesc_bf16_f32(C::kMmaM, BN, false);
            constexpr uint32_t kIdescPV = F8 ? ptx::idesc_e4m3_f32(BM, D, true)
                                             : ptx::idesc_bf16_f32(C::kMmaM, D, true);
            auto commit = [&](int i) {
                if constexpr (PAIR) ptx::mma_commit_pair(bar(i), 0x3);
                else ptx::mma_commit(bar(i));
            };
            int pv_done[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) pv_done[t] = 0;
            bool ok = true;
            // O_t (+)= P_t V_{s-1} (A = P_t from tensor memory) and S_t = Q_t K_s^T.
            auto issue_pv = [&](int t, int vst, bool first) {
                const uint32_t vbase = sbase + C::kVOff + vst * C::kSlotBytes;
                const uint64_t vdesc0 = ptx::sdesc_sw128(vbase, C::kVChunkBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < C::kPVSteps; ++kk) {
                    const uint64_t bdesc = ptx::sdesc_add(vdesc0, kk * C::kPVKeys * C::kRowBytes);
                    const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
                    const uint32_t a_tm = tmem + C::s_col(t) + kk * 8;
                    if constexpr (F8)
                        ptx::mma_ts_f8(tmem + C::o_col(t), a_tm, bdesc, kIdescPV, acc);
                    else if constexpr (PAIR)
                        ptx::mma_ts_pair(tmem + C::o_col(t), a_tm, bdesc, kIdescPV, acc);
                    else
                        ptx::mma_ts(tmem + C::o_col(t), a_tm, bdesc, kIdescPV, acc);
                }
            };
            auto issue_s = [&](int t, int kst) {
                const uint32_t qbase = sbase + C::kQOff + t * C::kQTileBytes;
                const uint32_t kbase = sbase + C::kKOff + kst * C::kSlotBytes;
                const uint64_t adesc0 = ptx::sdesc_sw128(qbase, 16, 1024);
                const uint64_t bdesc0 = ptx::sdesc_sw128(kbase, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    const uint32_t koff = (kk / 4) * C::kQChunkBytes + (kk % 4) * 32;
                    const uint32_t boff = (kk / 4) * C::kKChunkBytes + (kk % 4) * 32;
                    const uint64_t adesc = ptx::sdesc_add(adesc0, koff);
                    const uint64_t bdesc = ptx::sdesc_add(bdesc0, boff);
                    if constexpr (F8)
                        ptx::mma_ss_f8(tmem + C::s_col(t), adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
                    else if constexpr (PAIR)
                        ptx::mma_ss_pair(tmem + C::s_col(t), adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
                    else
                        ptx::mma_ss(tmem + C::s_col(t), adesc, bdesc, kIdescS, kk > 0 ? 1u : 0u);
                }
                commit(C::bSFull + t);
            };
            // Both tiles covering every block: the schedule without range
            // tests (each branch in this loop costs the tensor pipe: BF16
            // prefill 1.315 -> 1.289 ms; E4M3, once its first step was
            // peeled and each tile's Q had its own barrier, 1.108 -> 1.070 ms).
            // A causal tile 1 covers one block more than tile 0 (the
            // diagonal block of its own rows): walked from the last block
            // down (rev), tile 0 starts one step later; otherwise the same
            // loop runs up to tile 0's last step, then one step of tile 1's.
            // Under a sliding window tile 1 also starts one step later
            // (late1: the window's lower edge is one block later for its
            // rows), and its first S comes first in that step, as the slot
            // release rule of early_s expects.
            const int h0 = R[0].hi, h1 = R[1].hi;
            const int off0 = R[0].lo - lo;          // tile 0's first step (1 when rev)
            const int off1 = R[1].lo - lo;          // tile 1's first step (1 when late1)
            const bool late1 = !rev && early_s == lo + 1 && R[0].lo == lo && h0 > lo + 1;
            const bool uniform = !PAIR && (R[0].lo == lo || rev) && (R[1].lo == lo || late1) &&
                                 h1 == hi && (h0 == hi || h0 == hi - 1);
            if (uniform) {
                // step 0, peeled: S_t once Q_t and the first K block have
                // landed, for the tiles that start there (tile 1's Q is loaded
                // last, or first when rev)
                ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bStep), 0, abort_flag, err,
                                                          kSiteKFull));
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (!ok || R[t].lo != lo) continue;
                    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bQFull + t), 0, abort_flag,
                                                              err, kSiteQFull));
                    if (!ok) break;
                    ptx::tc_fence_after();
                    if (leader) issue_s(t, 0);
                    __syncwarp();
                }
                int s_first = lo + 1;
                if (rev && ok) {
                    // step 1, peeled: tile 0's first S, then tile 1's first
                    // P V product and its next S
                    constexpr int kst = 1 % NSK, vst = 0;
                    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bStep + kst), (1 / NSK) & 1,
                                                              abort_flag, err, kSiteKFull));
                    if (ok)
                        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bQFull), 0, abort_flag, err,
                                                                  kSiteQFull));
                    if (ok) {
                        ptx::tc_fence_after();
                        if (leader) issue_s(0, kst);
                        __syncwarp();
                        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bPFull + 1), 0, abort_flag,
                                                                  err, kSitePFull));
                    }
                    if (ok) {
                        ptx::tc_fence_after();
                        if (leader) {
                            issue_pv(1, vst, true);
                            issue_s(1, kst);                 // hi >= lo + 2 when rev
                        }
                        __syncwarp();
                    }
                    s_first = lo + 2;
                }
                if (late1 && ok) {
                    // step 1, peeled: tile 1's first S, then tile 0's first
                    // P V product and its next S
                    constexpr int kst = 1 % NSK, vst = 0;
                    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bStep + kst), (1 / NSK) & 1,
                                                              abort_flag, err, kSiteKFull));
                    if (ok)
                        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bQFull + 1), 0, abort_flag,
                                                                  err, kSiteQFull));
                    if (ok) {
                        ptx::tc_fence_after();
                        if (leader) issue_s(1, kst);
                        __syncwarp();
                        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bPFull), 0, abort_flag,
                                                                  err, kSitePFull));
                    }
                    if (ok) {
                        ptx::tc_fence_after();
                        if (leader) {
                            issue_pv(0, vst, true);
                            issue_s(0, kst);                 // h0 > lo + 1 when late1
                        }
                        __syncwarp();
                    }
                    s_first = lo + 2;
                }
                for (int s = s_first; ok && s <= h0; ++s) {
                    const int i = s - lo;
                    const int kst = i % NSK;
                    const int vst = (i + NSV - 1) % NSV;
                    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bStep + kst), (i / NSK) & 1,
                                                              abort_flag, err, kSiteKFull));
                    if (!ok) break;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const int pi = i - 1 - (t == 0 ? off0 : off1);   // tile t's P hand-off index
                        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bPFull + t), pi & 1,
                                                                  abort_flag, err, kSitePFull));
                        if (!ok) break;
                        ptx::tc_fence_after();
                        if (leader) {
                            issue_pv(t, vst, pi == 0);
                            if (s == R[t].hi) commit(C::bODone + t);
                        }
                        __syncwarp();
                        if (s < R[t].hi) {
                            if (leader) issue_s(t, kst);
                            __syncwarp();
                        }
                    }
                    if (!ok) break;
                }
                if (ok && h0 < hi) {
                    // tile 1's last P V product (step hi)
                    const int i = hi - lo;
                    ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bStep + i % NSK), (i / NSK) & 1,
                                                              abort_flag, err, kSiteKFull));
                    if (ok)
                        ok = __all_sync(0xffffffffu, wait_bounded(bar(C::bPFull + 1),
                                                                  (i - 1 - off1) & 1, abort_flag,
                                                                  err, kSitePFull));
                    if (ok) {
                        ptx::tc_fence_after();
                        if (leader) {
                            issue_pv(1, (i + NSV - 1) % NSV, i - 1 - off1 == 0);
                            commit(C::bODone + 1);
                        }
                        __syncwarp();
                    }
                }
            }
            for (int s = lo; ok && !uniform && s <= hi; ++s) {
                const int i = s - lo;
                const int kst = i % NSK;                       // K slot of block s = step barrier
                const uint32_t kph = (i / NSK) & 1;
                const int vst = (i + NSV - 1) % NSV;           // V slot of block s - 1
                // The step barrier (K_s and V_{s-1} landed) is waited right
                // before the step's first MMA, and once per step in any case.
                bool kv_ready = false;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (s - 1 >= R[t].lo && s - 1 < R[t].hi) {
                        // O_t (+)= P_t V_{s-1} once the softmax has stored P_t.
                        if (!kv_ready) {
                            ok = __all_sync(0xffffffffu,
                                            wait_bounded<PAIR>(bar(C::bStep + kst), kph, abort_flag,
                                                               err, kSiteKFull));
                            if (!ok) break;
                            kv_ready = true;
                        }
                        ok = __all_sync(0xffffffffu,
                                        wait_bounded<PAIR>(bar(C::bPFull + t), pv_done[t] & 1,
                                                           abort_flag, err, kSitePFull));
                        if (!ok) break;
                        ptx::tc_fence_after();
                        if (leader) {
                            issue_pv(t, vst, pv_done[t] == 0);
                            if (s - 1 == R[t].hi - 1) commit(C::bODone + t);
                        }
                        __syncwarp();
                        ++pv_done[t];
                    }
                    if (s < hi && s >= R[t].lo && s < R[t].hi) {
                        // S_t = Q_t K_s^T (the tile's first: once its Q has landed)
                        if (!kv_ready) {
                            ok = __all_sync(0xffffffffu,
                                            wait_bounded<PAIR>(bar(C::bStep + kst), kph, abort_flag,
                                                               err, kSiteKFull));
                            if (!ok) break;
                            ptx::tc_fence_after();
                            kv_ready = true;
                        }
                        if (s == R[t].lo) {
                            ok = __all_sync(0xffffffffu, wait_bounded<PAIR>(bar(C::bQFull + t), 0,
                                                                            abort_flag, err,
                                                                            kSiteQFull));
                            if (!ok) break;
                            ptx::tc_fence_after();
                        }
                        if (leader) issue_s(t, kst);
                        __syncwarp();
                    }
                }
                if (!ok) break;
                if (!kv_ready)
                    ok = __all_sync(0xffffffffu, wait_bounded<PAIR>(bar(C::bStep + kst), kph,
                                                                    abort_flag, err, kSiteKFull));
                if (!ok) break;
                // K_s and V_{s-1} are released by the softmax (no commit here:
                // each commit costs the issue stream a few hundred cycles).
            }
            // Every MMA issued above completes before tensor memory is freed.
            if (leader) commit(C::bDrain);
            __syncwarp();
        }
        if (lo < hi) wait_bounded<PAIR>(bar(C::bDrain), 0, nullptr, err, kSiteDrain);
    } else {
        // ------------------------------------------------ softmax, epilogue
        const int t = warp / 4, wq = warp % 4;
        const Range Rt = (t == 0) ? R[0] : R[1];
        const int r = wq * 32 + lane;
        const int row_first = own_row(t);
        const int row = row_first + r;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + C::s_col(t);
        const uint32_t o_addr = tmem + lane_base + C::o_col(t);
        // m_use: the reference the row's P, l and A are currently scaled to.
        // It moves only when a block's max exceeds it by more than kTau
        // (log2 units), so P <= 2^kTau and A is rescaled rarely; the final
        // A / l and lse = m_use + log l are exact for any reference.
        float m_use = -INFINITY, l = 0.f;
        int c = 0;
        bool ok = true;
        const float2 c2 = make_float2(scale_log2, scale_log2);
        for (int j = Rt.lo; j < Rt.hi; ++j, ++c) {
            const bool got = wait_bounded<PAIR>(bar(C::bSFull + t), c & 1, abort_flag, err,
                                                kSiteSFull);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            // Release K_j and V_{j-1}. In issue order PV_0(j-1), S_0(j),
            // PV_1(j-1), S_1(j), the last MMA of step j that reads either is
            // the S product of the last tile covering block j (tile 1 on its
            // range, tile 0 on the blocks before it: the ranges are contiguous
            // and tile 1's ends last), and its completion implies every
            // earlier one. At tile 1's early first block the order is S_1(j),
            // PV_0(j-1), S_0(j), so tile 0 releases it. Nobody waits for the
            // last blocks' releases.
            const int releaser = (j == early_s) ? 0
                                 : (j >= R[NT - 1].lo && j < R[NT - 1].hi) ? NT - 1 : 0;
            if (wq == 0 && lane == 0 && t == releaser) {
                const int ii = j - lo;
                ptx::mbar_arrive(bar(C::bKEmpty + ii % NSK));
                if (ii > 0) ptx::mbar_arrive(bar(C::bVEmpty + (ii - 1) % NSV));
            }
            ptx::tc_fence_after();
            uint32_t sr[BN];
            ptx::tmem_ld32x32b_x128(s_addr, sr);
            const int kb = blk(j) * BN;
            if (block_needs_mask(kb, row_first, Lk, causal, windowed, window)) {
                // the row's visible keys in this block are one interval
                // [kb + a, kb + e): one unsigned comparison per key
                int a = 0, e = min(BN, Lk - kb);
                if (causal) e = min(e, row + 1 - kb);
                if (windowed) a = max(0, row - window + 1 - kb);
                const unsigned span = static_cast<unsigned>(max(e - a, 0));
#pragma unroll
                for (int kk = 0; kk < BN; ++kk)
                    if (static_cast<unsigned>(kk - a) >= span) sr[kk] = __float_as_uint(-INFINITY);
            }
            // row max: four independent chains of three-input max
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int kk = 0; kk < BN; kk += 8) {
                mx0 = ptx::max3(mx0, __uint_as_float(sr[kk]), __uint_as_float(sr[kk + 1]));
                mx1 = ptx::max3(mx1, __uint_as_float(sr[kk + 2]), __uint_as_float(sr[kk + 3]));
                mx2 = ptx::max3(mx2, __uint_as_float(sr[kk + 4]), __uint_as_float(sr[kk + 5]));
                mx3 = ptx::max3(mx3, __uint_as_float(sr[kk + 6]), __uint_as_float(sr[kk + 7]));
            }
            const float m_blk = ptx::max3(mx0, mx1, fmaxf(mx2, mx3)) * scale_log2;
            const bool need = m_blk > m_use + kTau;          // false while the block is empty
            const float m_next = need ? m_blk : m_use;
            const float m_ref = (m_next == -INFINITY) ? 0.f : m_next;   // the P2 guard
            const float alpha = need ? ptx::ex2(m_use - m_ref) : 1.f;
            // P = exp2(S * scale * log2e - m_ref), one 64-key half at a time
            // (fewer live registers): BF16 pairs into tensor memory over S.
            const float2 nm2 = make_float2(-m_ref, -m_ref);
            float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // BF16: two stores of 16 columns (32 keys each) per half;
                // E4M3: one store of 16 columns (64 keys) per half.
                uint32_t pk8[16];
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int kp = 0; kp < 16; kp += 4) {
                        float2 p[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int kk = half * (BN / 2) + q4 * 32 + 2 * (kp + u);
                            const float2 x = __ffma2_rn(
                                make_float2(__uint_as_float(sr[kk]), __uint_as_float(sr[kk + 1])),
                                c2, nm2);
                            if (soft_pair<F8>(kp + u))
                                p[u] = soft_exp2x2(x);
                            else
                                p[u] = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
                            if constexpr (!F8) pk[kp + u] = pack_bf16x2(p[u].x, p[u].y);
                        }
                        if constexpr (F8) {
                            pk8[q4 * 8 + kp / 2] = ptx::pack_e4m3x4(p[0].x, p[0].y, p[1].x, p[1].y);
                            pk8[q4 * 8 + kp / 2 + 1] =
                                ptx::pack_e4m3x4(p[2].x, p[2].y, p[3].x, p[3].y);
                        }
                        acc0 = __fadd2_rn(acc0, p[0]);
                        acc1 = __fadd2_rn(acc1, p[1]);
                        acc2 = __fadd2_rn(acc2, p[2]);
                        acc3 = __fadd2_rn(acc3, p[3]);
                    }
                    if constexpr (!F8)
                        ptx::tmem_st32x32b_x16(s_addr + half * C::kPHalfCols + q4 * 16, pk);
                }
                if constexpr (F8) ptx::tmem_st32x32b_x16(s_addr + half * C::kPHalfCols, pk8);
                // Before the first P V product of this block: A <- diag(alpha) A,
                // only for warps where some row moved its reference (rows that
                // did not move multiply by exactly 1). Done here, after the
                // first half of the scores is consumed, to keep registers low.
                if (half == 0 && __any_sync(0xffffffffu, need && m_use != -INFINITY)) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t ov[32];
                        ptx::tmem_ld32x32b_x32(o_addr + cc * 32, ov);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 r = __fmul2_rn(
                                make_float2(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])),
                                make_float2(alpha, alpha));
                            ov[e] = __float_as_uint(r.x);
                            ov[e + 1] = __float_as_uint(r.y);
                        }
                        ptx::tmem_st32x32b_x32(o_addr + cc * 32, ov);
                    }
                }
            }
            // both halves of P (and any rescale of A) stored: hand P over
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) ptx::mbar_arrive_cluster(lead_bar(C::bPFull + t));
                else ptx::mbar_arrive(bar(C::bPFull + t));
            }
            const float2 a01 = __fadd2_rn(acc0, acc1), a23 = __fadd2_rn(acc2, acc3);
            const float2 asum = __fadd2_rn(a01, a23);
            l = fmaf(l, alpha, asum.x + asum.y);
            m_use = m_next;
        }
        if (ok && c > 0) {
            const bool got = wait_bounded<PAIR>(bar(C::bODone + t), 0, abort_flag, err, kSiteODone);
            ok = __all_sync(0xffffffffu, got);
            ptx::tc_fence_after();
        }
        const bool have = ok && c > 0;
        const float inv_l = (l > 0.f) ? o_mul / l : 0.f;
        // O_t goes through tile t's Q buffer (free once O_t is final: every
        // S_t product was issued before the last P_t V one) in the
        // 128-byte-swizzled layout Q arrived in -- 16-byte chunk j of row r
        // at j ^ (r % 8), so a warp's stores hit every bank once per
        // wavefront -- and leaves in one TMA store per 64 head dims, each
        // issued as soon as its chunk is staged (the TMA reads shared memory
        // at about 40 bytes per cycle, so the first read overlaps the second
        // chunk's conversion). The buffer holds all of a BF16 O tile; with
        // E4M3 inputs (a Q tile of half the bytes) O goes in two passes of
        // 64 head dims.
        const uint32_t obuf = sbase + C::kQOff + t * C::kQTileBytes;
        constexpr uint32_t kOChunkBytes = BM * 128;                 // 64 BF16 head dims
        constexpr int kOChunks = D / 64;
        constexpr int kOPerPass = static_cast<int>(C::kQTileBytes / kOChunkBytes);
        static_assert(kOPerPass >= 1 && kOChunks % kOPerPass == 0, "O passes");
        const bool issuer = wq == 0 && lane == 0 && row_first < Nq;
#pragma unroll
        for (int oc = 0; oc < kOChunks; ++oc) {                     // 64 head dims at a time
            uint32_t ov[64];
            if (have) {
                ptx::tmem_ld32x32b_x64(o_addr + oc * 64, ov);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) ov[e] = 0u;
            }
            const uint32_t rbase = obuf + (oc % kOPerPass) * kOChunkBytes + r * 128;
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) {                           // 16-byte chunks of the row
                uint32_t pw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pw[e] = pack_bf16x2(__uint_as_float(ov[8 * jc + 2 * e]) * inv_l,
                                        __uint_as_float(ov[8 * jc + 2 * e + 1]) * inv_l);
                ptx::st_shared_v4(rbase + ((jc ^ (r & 7)) << 4), pw[0], pw[1], pw[2], pw[3]);
            }
            // each 64-dim chunk leaves as soon as it is in shared memory (the
            // TMA reads it while the next chunk is converted)
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1 + t, 4 * 32);                 // the tile's four warps
            if (issuer) {
                ptx::tma_store_3d(&tm_o, obuf + (oc % kOPerPass) * kOChunkBytes, oc * 64, row_first,
                                  bh);
                ptx::bulk_commit_group();
            }
            if ((oc + 1) % kOPerPass == 0) {
                if (oc + 1 < kOChunks) {
                    // the buffer is reused by the next pass once the copy has read it
                    if (issuer) ptx::bulk_wait_read_all();
                    ptx::named_bar_sync(1 + t, 4 * 32);
                }
            }
        }
        if (lse != nullptr && row < Nq)
            lse[static_cast<long long>(bh) * Nq + row] =
                (l > 0.f) ? (m_use + log2f(l)) * kLn2 : -INFINITY;
        if (issuer) ptx::bulk_wait_read_all();   // the buffer outlives the copy's reads
    }

    ptx::tc_fence_before();
    if constexpr (PAIR) {
        // Neither CTA leaves while the other may still signal its barriers
        // or the pair's MMAs read its shared and tensor memory.
        ptx::cluster_arrive_release();
        ptx::cluster_wait_acquire();
    } else {
        __syncthreads();
    }
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, kTmemCols);
        else ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool F8, bool PAIR>
cudaError_t launch_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, const CUtensorMap& to, float scale_log2, float o_mul,
                     cudaStream_t stream) {
    using C = Cfg<D, F8, PAIR>;
    static int configured_device = -1;   // attribute is per device; set once per device seen
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(fwd_sm103_kernel<D, F8, PAIR>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int units = (a.Nq + C::kMmaM * NT - 1) / (C::kMmaM * NT);
    dim3 grid(units * C::kCtas, a.H, a.B);
    // Causal or windowed: longest units first within groups of heads whose
    // K and V together take about a quarter of L2 (32 MiB), or half of it
    // (64 MiB) under a sliding window, where a CTA reads only a window's
    // worth of K and V (masked B8 H16 4096^2: 0.1653 -> 0.1606 ms, the
    // longest-first order balancing over twice the heads; causal B2 H32
    // 8192^2 kept its time with half but re-read 45 MB of K and V).
    int group_heads = 0;
    if (a.mask_kind & (kMaskCausal | kMaskWindow)) {
        const long long nbh = static_cast<long long>(a.B) * a.H;
        const long long kv_head = 2LL * a.Nk * a.d * C::kElem;
        const long long budget = (a.mask_kind & kMaskWindow) ? (64LL << 20) : (32LL << 20);
        const long long g = std::max(1LL, budget / std::max(kv_head, 1LL));
        group_heads = static_cast<int>(std::min(g, nbh));
        // the kernel computes this order in 32-bit arithmetic
        if (static_cast<long long>(grid.x) * grid.y * grid.z > INT_MAX) group_heads = 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if constexpr (PAIR) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fwd_sm103_kernel<D, F8, PAIR>, tq, tk, tv, to,
                              static_cast<__nv_bfloat16*>(a.o), a.lse, a.H, a.Nq, a.Nk,
                              scale_log2, o_mul, a.mask_kind, a.window, a.seqlens_k, a.err,
                              group_heads);
}

}  // namespace

// pair: the CTA-pair kernel (d = 128; tk then has boxes of 64 keys).
cudaError_t launch_fwd_sm103_maps(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& to, bool pair,
                                  cudaStream_t stream) {
    const float sl2 = a.scale * kLog2e;
    if (a.d == 64) return launch_d<64, false, false>(a, tq, tk, tv, to, sl2, 1.f, stream);
    return pair ? launch_d<128, false, true>(a, tq, tk, tv, to, sl2, 1.f, stream)
                : launch_d<128, false, false>(a, tq, tk, tv, to, sl2, 1.f, stream);
}

// E4M3 inputs, d = 128: the score scale folds the Q and K dequantisation
// factors, and the output multiplier is V's factor (O = descale_v A / l).
cudaError_t launch_fwd_fp8_maps(const FwdArgs& a, float descale_q, float descale_k,
                                float descale_v, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to,
                                cudaStream_t stream) {
    const float sl2 = a.scale * descale_q * descale_k * kLog2e;
    return launch_d<128, true, false>(a, tq, tk, tv, to, sl2, descale_v, stream);
}

}  // namespace attn
