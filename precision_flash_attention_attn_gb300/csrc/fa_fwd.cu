// Flash-attention forward for sm_103a: tiled online safe softmax in three
// modes (baseline, stabilised, FP32 output), BF16 Q/K/V, FP32 TMEM
// accumulators.
//
// Computes, per row i of a (batch, head):  S = Q K^T (raw scores),
// Pbar = exp(alpha*S - m), Obar = Pbar V, O = Obar / rowsum(Pbar),
// LSE = m + ln rowsum(Pbar)   ("Why Low-Precision Transformer Training Fails:
// An Analysis on Flash Attention", section 3.4.4, safe-softmax equations).
// The shift m is the running row max (modes 0, 2) or the stabilised shift of
// section 3.4.5 (mode 1): with running max M and running count C of keys equal
// to M, m = beta*M if M > 0 and C > 1, 0 if M < 0 and C > 1, else M (ties are
// exact equality of FP32 raw scores, eps = 0).
//
// One CTA owns NQ (1 or 2) consecutive 128-row query tiles of one (batch,
// head) and streams 128-key K/V tiles shared by them.  Warp roles:
//   warps 4t..4t+3  softmax of query tile t: thread r owns row r (TMEM lane
//              r).  Reads S from TMEM (and frees it at once), masks, reduces
//              the row max and tie count, updates the shift, waits for the
//              previous Pbar V product, rescales the O accumulator in TMEM
//              when the shift changed, exponentiates (ex2) while writing BF16
//              Pbar to tensor memory, and finally normalises and stores O and
//              the LSE.
//   warp 4*NQ  TMA producer: the Q tiles once, then K and V tiles in a ring.
//   warp 4*NQ+1+t  MMA issuer of query tile t: S_t = Q_t K_j^T into the
//              tile's TMEM S buffer as soon as the softmax has read the
//              previous S, then O_t += Pbar_t V_{j-1} (tcgen05.mma kind::f16;
//              Q, K, V from shared memory, Pbar from tensor memory).  One
//              issuer per tile keeps the two tiles' chains independent: each
//              softmax warpgroup waits only for its own MMAs, and the tensor
//              core interleaves the two tiles' work.  A K/V stage is refilled
//              once every tile that reads it has finished its PV product.
// With two query tiles the CTA has three warpgroups; the producer/MMA
// warpgroup hands registers to the two softmax warpgroups (setmaxnreg).
// TMEM columns: S_t at 128*t, O_t at 128*NQ + d*t, Pbar_t (BF16 pairs) after
// the O accumulators, 64 columns each.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

template <int D, int MODE, int NQ>
struct FwdLayout {
    static constexpr int kTileBytes = kBlockM * D * 2;  // 128 rows x D BF16
    static constexpr int kPBytes = kBlockM * kBlockN * 2;
    // Pbar lives in TMEM (the A operand of Pbar V).  The FP32-output mode also
    // feeds a lo part (Pbar = hi + lo, both BF16): in TMEM where columns allow,
    // otherwise in shared memory.
    static constexpr bool kLoInTmem = (MODE == 2) && (NQ * (128 + D + 64 + 64) <= 512);
    static constexpr bool kLoInSmem = (MODE == 2) && !kLoInTmem;
    // Q is double-buffered where shared memory allows, so the next work
    // item's Q lands while the current one is still being multiplied.
    static constexpr int kQBufs = (D == 64) ? 2 : 1;
    static constexpr int kStages = (D == 64) ? (kLoInSmem ? 3 : 4) : 3;
    static constexpr int kQ = 0;                                  // [kQBufs][NQ]
    static constexpr int kK = kQ + kQBufs * NQ * kTileBytes;      // [kStages]
    static constexpr int kV = kK + kStages * kTileBytes;          // [kStages]
    static constexpr int kPLo = kV + kStages * kTileBytes;        // [NQ], mode 2 without TMEM room
    // With d = 64 the epilogue stages O in shared memory and writes it with
    // TMA stores (row-per-thread global stores would scatter 32 rows per
    // warp instruction).  The FP32-output mode stages O in its lo buffer,
    // which is free between the item's last Pbar V and the next item's first
    // Pbar; the other modes have a buffer of their own.
    static constexpr bool kTmaStoreO = (D == 64);
    static constexpr int kOStageBytes = kBlockM * D * 2;
    static constexpr int kOStage = kPLo + (kLoInSmem ? NQ * kPBytes : 0);  // [NQ], modes 0 and 1
    static constexpr int kBar = kOStage + ((kTmaStoreO && MODE != 2) ? NQ * kOStageBytes : 0);
    static_assert(!kTmaStoreO || MODE != 2 || kLoInSmem, "FP32 O staging uses the lo buffer");
    // barriers
    static constexpr int kQFull = 0;                     // [kQBufs]
    static constexpr int kQEmpty = kQFull + kQBufs;      // [kQBufs], one arrival per tile
    static constexpr int kKFull = kQEmpty + kQBufs;      // [kStages]
    static constexpr int kVFull = kKFull + kStages;      // [kStages]
    static constexpr int kKVEmpty = kVFull + kStages;    // [NQ][kStages]
    static constexpr int kSFull = kKVEmpty + NQ * kStages;  // [NQ]
    static constexpr int kSEmpty = kSFull + NQ;        // [NQ]
    static constexpr int kPFull = kSEmpty + NQ;        // [NQ]
    static constexpr int kODone = kPFull + NQ;         // [NQ]
    static constexpr int kOFree = kODone + NQ;         // [NQ]: O read out by the epilogue
    static constexpr int kOStaged = kOFree + NQ;       // [NQ]: O rows written to the staging buffer
    static constexpr int kStageFree = kOStaged + NQ;   // [NQ]: previous TMA store has read the buffer
    static constexpr int kDrain = kStageFree + NQ;     // [NQ]
    static constexpr int kNumBars = kDrain + NQ;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kBytes = kTmemSlot + 16;
    static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
    static constexpr uint32_t kTmemUsed = NQ * (128 + D + 64) + (kLoInTmem ? NQ * 64 : 0);
    static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static_assert(kTmemUsed <= 512, "TMEM budget");
    static constexpr uint32_t kSCol = 0;                   // [NQ] x 128: S (FP32)
    static constexpr uint32_t kOCol = 128 * NQ;            // [NQ] x D: O accumulator
    static constexpr uint32_t kPCol = kOCol + NQ * D;      // [NQ] x 64: Pbar (BF16 pairs)
    static constexpr uint32_t kPLoCol = kPCol + NQ * 64;   // [NQ] x 64: Pbar lo (mode 2, if room)
    // softmax warpgroups, then producer + one MMA warp per tile (padded to a
    // whole warpgroup when registers are rebalanced)
    static constexpr int kThreads = NQ == 2 ? 384 : 192;
    // register budgets with two tiles (2 x 128 x softmax + 128 x other =
    // 384 x 168): the FP32-output mode's MMA warps issue the lo products too
    static constexpr uint32_t kRegsSoftmax = MODE == 2 ? 200 : 216;
    static constexpr uint32_t kRegsOther = MODE == 2 ? 104 : 72;
    static_assert(NQ != 2 || 256 * kRegsSoftmax + 128 * kRegsOther == 384 * 168, "register split");
    static_assert(kAlloc <= 232448, "shared memory budget");
};

struct FwdParams {
    void* o;
    float* lse;
    int32_t* tie_count;
    int32_t* p_one;
    int BH, N;
    int n_cq;     // query-tile groups (of NQ tiles) per (batch, head)
    int n_items;  // BHon * n_cq work items
    float scale_log2;
    float beta;   // mode 1: shift factor of rows with a positive repeated maximum
    int* status;
    int test_withhold_k;  // test hook (see FwdArgs)
    const float* shift;   // mode 1, nullable: fixed per-row shift (see FwdArgs)
    const int32_t* rs_in; // statistics variant, nullable: tie counts to report
    uint64_t head_mask;   // heads h (bit h) this launch computes
    int H;
    int Hon, BHon;        // heads in head_mask (of H), batch x those heads
    RowLayout lay;        // q, k, v, o rows (the tensor maps are 4-D: column, row, head, batch)
};

// Work items are (query-tile group, batch-head) pairs, numbered longest first
// (largest causal group index first).  CTA c takes items in a snake order over
// rounds of gridDim.x: round r visits c on even rounds and gridDim.x-1-c on
// odd ones, which balances the causal work nearly as well as greedy longest-
// processing-time scheduling.
// Whether the maximum tm of a tile of kBlockN scores s[c] occurs at least
// twice, given mx[e] = max of s[c] over c = e (mod 8).  Two distinct keys
// differ in c mod 8 or, if not, in c div 8, so it does exactly when two of
// the mod-8 chain maxima, or two of the maxima of the 16 blocks of 8
// consecutive keys, equal tm.
__device__ __forceinline__ bool tile_max_repeats(const float (&s)[kBlockN], const float (&mx)[8], float tm) {
    int na = 0, nb = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) na += (mx[e] == tm) ? 1 : 0;
#pragma unroll
    for (int b = 0; b < kBlockN / 8; ++b) {
        const float* v8 = &s[8 * b];
        const float bm = fmax3(fmax3(v8[0], v8[1], v8[2]), fmax3(v8[3], v8[4], v8[5]), fmaxf(v8[6], v8[7]));
        nb += (bm == tm) ? 1 : 0;
    }
    return na >= 2 || nb >= 2;
}

// Position of the k-th (from 0) set bit of m; m has more than k set bits.
__device__ __forceinline__ int nth_set_bit(uint64_t m, int k) {
    uint32_t w = static_cast<uint32_t>(m);
    int base = 0;
    const int lo = __popc(w);
    if (k >= lo) {
        k -= lo;
        w = static_cast<uint32_t>(m >> 32);
        base = 32;
    }
    for (int i = 0; i < k; ++i) w &= w - 1u;  // drop the k lowest set bits
    return base + __ffs(static_cast<int>(w)) - 1;
}

__device__ __forceinline__ int fwd_item(int r) {
    const int G = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    return r * G + ((r & 1) ? G - 1 - c : c);
}

template <int D, int MODE, bool CAUSAL, bool STATS, int NQ>
__global__ void __launch_bounds__(FwdLayout<D, MODE, NQ>::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
    using L = FwdLayout<D, MODE, NQ>;
    constexpr int S = L::kStages;
    constexpr int QB = L::kQBufs;
    constexpr int kProducerWarp = 4 * NQ;
    constexpr int kMmaWarp0 = 4 * NQ + 1;  // MMA issuer of tile t: warp kMmaWarp0 + t
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + L::kBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_ktiles_all = (p.N + kBlockN - 1) / kBlockN;
    // Work item -> (batch-head, group); per query tile t of the group: first
    // row and number of key tiles it visits (0: the tile lies past N).
    // Only the heads of this launch's set are items: item x of a group is
    // head number x % Hon of the set (in increasing h) of batch x / Hon.
    auto item_bh = [&](int it) {
        const int x = it % p.BHon;
        if (p.Hon == p.H) return x;
        return (x / p.Hon) * p.H + nth_set_bit(p.head_mask, x % p.Hon);
    };
    auto item_cq = [&](int it) { return p.n_cq - 1 - it / p.BHon; };
    auto tile_q0 = [&](int cq, int t) { return (cq * NQ + t) * kBlockM; };
    auto tile_nkt = [&](int it, int t) {
        const int qt = item_cq(it) * NQ + t;
        if (qt * kBlockM >= p.N) return 0;
        return CAUSAL ? (qt + 1 < n_ktiles_all ? qt + 1 : n_ktiles_all) : n_ktiles_all;
    };
    auto item_nkt = [&](int it) {
        int n = 0;
#pragma unroll
        for (int t = 0; t < NQ; ++t) n = tile_nkt(it, t) > n ? tile_nkt(it, t) : n;
        return n;
    };

    if (threadIdx.x == 0) {
        for (int b = 0; b < QB; ++b) {
            mbar_init(bar(L::kQFull + b), 1);
            mbar_init(bar(L::kQEmpty + b), NQ);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(L::kKFull + s), 1);
            mbar_init(bar(L::kVFull + s), 1);
        }
        for (int t = 0; t < NQ; ++t) {
            for (int s = 0; s < S; ++s) mbar_init(bar(L::kKVEmpty + t * S + s), 1);
            mbar_init(bar(L::kSFull + t), 1);
            mbar_init(bar(L::kSEmpty + t), 128);
            mbar_init(bar(L::kPFull + t), 128);
            mbar_init(bar(L::kODone + t), 1);
            mbar_init(bar(L::kOFree + t), 128);
            mbar_init(bar(L::kOStaged + t), 128);
            mbar_init(bar(L::kStageFree + t), 1);
            mbar_init(bar(L::kDrain + t), 1);
        }
        fence_mbar_init();
    }
    if (warp == kMmaWarp0) {
        tmem_alloc(sb + L::kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    // Nothing above reads or writes global memory, so under programmatic
    // dependent launch all of it overlaps the previous kernel in the stream.
    griddep_wait();
    // The next kernel may be launched now: its CTAs take the SMs this grid's
    // CTAs leave (the causal items are unequal, so some leave early) and
    // start on work that does not depend on this grid (the backward's first
    // kernel loads dO); its griddepcontrol.wait still waits for all of this
    // grid and its memory operations.
    griddep_launch_dependents();

    if (warp >= kProducerWarp) {
        if (NQ == 2) regs_dec<L::kRegsOther>();
        if (warp == kProducerWarp) {
            // ------------------------------------------------------ TMA producer
            // Streams every item's Q tiles and K/V tiles through the rings,
            // running ahead into the next item as far as the buffers allow.
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                bool ok = true;
                int g = 0;  // K/V tiles issued so far (all items)
                int n = 0;  // items started
                for (int r = 0; ok; ++r, ++n) {
                    const int it = fwd_item(r);
                    if (it >= p.n_items) break;
                    const int bh = item_bh(it), cq = item_cq(it);
                    const int hh = bh % p.H, bb = bh / p.H;  // head and batch of the tile coordinates
                    const int qb = n % QB;
                    const uint32_t uq = static_cast<uint32_t>(n / QB);
                    // the Q buffer is free once both tiles' last S of item n - QB is done
                    if (n >= QB) ok = mbar_wait(bar(L::kQEmpty + qb), (uq - 1) & 1u, p.status);
                    if (!ok) break;
                    int n_active = 0;
                    for (int t = 0; t < NQ; ++t) n_active += tile_nkt(it, t) > 0 ? 1 : 0;
                    mbar_arrive_expect_tx(bar(L::kQFull + qb), L::kTileBytes * n_active);
                    for (int t = 0; t < NQ; ++t) {
                        if (tile_nkt(it, t) == 0) continue;
                        for (int b = 0; b < D / 64; ++b)
                            tma_load_rows(sb + L::kQ + (qb * NQ + t) * L::kTileBytes + b * 16384, &tm_q,
                                        bar(L::kQFull + qb), b * 64, tile_q0(cq, t), hh, bb, p.lay.head_inner);
                    }
                    const int n_kt = item_nkt(it);
                    for (int j = 0; j < n_kt; ++j, ++g) {
                        const int s = g % S;
                        const uint32_t u = static_cast<uint32_t>(g / S);
                        // At the start every CTA asks for its Q tiles and all K/V
                        // stages at once; the first K tile, which the first S
                        // needs, then queues behind the rest in DRAM.  The later
                        // stages are issued once it has landed.
                        if (g == 1 && !(p.test_withhold_k && blockIdx.x == 0))
                            ok = mbar_wait(bar(L::kKFull), 0u, p.status);
                        // stage s is free once every tile has released round u-1
                        if (ok && g >= S)
                            for (int t = 0; t < NQ && ok; ++t)
                                ok = mbar_wait(bar(L::kKVEmpty + t * S + s), (u - 1) & 1u, p.status);
                        if (!ok) break;
                        // test hook: CTA 0 never loads its first K tile, so the
                        // waits on it run out (nothing is left in flight)
                        const bool withhold = p.test_withhold_k && blockIdx.x == 0 && g == 0;
                        if (!withhold) {
                            mbar_arrive_expect_tx(bar(L::kKFull + s), L::kTileBytes);
                            for (int b = 0; b < D / 64; ++b)
                                tma_load_rows(sb + L::kK + s * L::kTileBytes + b * 16384, &tm_k, bar(L::kKFull + s),
                                            b * 64, j * kBlockN, hh, bb, p.lay.head_inner);
                        }
                        mbar_arrive_expect_tx(bar(L::kVFull + s), L::kTileBytes);
                        for (int b = 0; b < D / 64; ++b)
                            tma_load_rows(sb + L::kV + s * L::kTileBytes + b * 16384, &tm_v, bar(L::kVFull + s),
                                        b * 64, j * kBlockN, hh, bb, p.lay.head_inner);
                    }
                }
                // Every copy this thread issued must have landed before the CTA
                // may exit (normally long since true).
                for (int m = n - QB > 0 ? n - QB : 0; m < n; ++m)
                    mbar_wait(bar(L::kQFull + m % QB), static_cast<uint32_t>(m / QB) & 1u, p.status);
                for (int h = g - S > 0 ? g - S : 0; h < g; ++h) {
                    const uint32_t u = static_cast<uint32_t>(h / S);
                    mbar_wait(bar(L::kKFull + h % S), u & 1u, p.status);
                    mbar_wait(bar(L::kVFull + h % S), u & 1u, p.status);
                }
            }
        } else if (warp < kMmaWarp0 + NQ) {
            // ------------------------------------------ MMA issuer of query tile t
            // The whole warp runs the loop and waits; one elected lane issues each
            // group of MMAs together with the commits that track them.  Per item:
            // S(0), then S(j) and Pbar V(j-1) alternately, then Pbar V(last).
            const int t = warp - kMmaWarp0;
            constexpr uint32_t kIdS = idesc_bf16(kBlockM, kBlockN, false, false);
            constexpr uint32_t kIdPV = idesc_bf16(kBlockM, D, false, true);
            const uint32_t s_acc = tmem + L::kSCol + t * 128;
            const uint32_t o_acc = tmem + L::kOCol + t * D;
            const uint32_t p_tm = tmem + L::kPCol + t * 64;
            const uint32_t plo_tm = tmem + L::kPLoCol + t * 64;
            auto wait_all = [&](uint32_t b, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, p.status));
            };
            bool ok = true;
            bool issued = false;
            int g = 0;   // K/V ring position of the current item's first tile
            int cs = 0;  // S (and Pbar) products of this tile so far, all items
            int e = 0;   // items this tile has finished (epilogues)
            // Pbar V for local key tile jj whose Pbar is number c of this tile
            auto issue_pv = [&](int jj, int c) {
                const int s = (g + jj) % S;
                const uint32_t u = static_cast<uint32_t>((g + jj) / S);
                ok = ok && wait_all(bar(L::kVFull + s), u & 1u);
                ok = ok && wait_all(bar(L::kPFull + t), static_cast<uint32_t>(c) & 1u);
                // the first product of an item overwrites O: the previous
                // item's epilogue must have read it out
                if (jj == 0 && e >= 1) ok = ok && wait_all(bar(L::kOFree + t), static_cast<uint32_t>(e - 1) & 1u);
                if (!ok) return;
                tc_fence_after();
                const uint32_t v_sm = sb + L::kV + s * L::kTileBytes;
                if (elect_one()) {
                    // A = Pbar from TMEM: 16 keys (8 columns) per MMA step
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)
                        mma_bf16_ts(o_acc, p_tm + kk * 8, sdesc_sw128(v_sm + kk * 2048, 16384, 1024), kIdPV,
                                    (jj > 0 || kk > 0) ? 1u : 0u);
                    if (L::kLoInTmem) {
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk)
                            mma_bf16_ts(o_acc, plo_tm + kk * 8, sdesc_sw128(v_sm + kk * 2048, 16384, 1024), kIdPV,
                                        1u);
                    } else if (L::kLoInSmem) {
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk) {
                            const uint64_t a = sdesc_sw128(
                                sb + L::kPLo + t * L::kPBytes + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                            mma_bf16_ss(o_acc, a, sdesc_sw128(v_sm + kk * 2048, 16384, 1024), kIdPV, 1u);
                        }
                    }
                    mma_commit(bar(L::kODone + t));
                    mma_commit(bar(L::kKVEmpty + t * S + s));
                }
                __syncwarp();
            };
            for (int r = 0, n = 0; ok; ++r, ++n) {
                const int it = fwd_item(r);
                if (it >= p.n_items) break;
                const int nkt = tile_nkt(it, t);
                const int n_kt = item_nkt(it);
                const int qb = n % QB;
                const uint32_t q_sm = sb + L::kQ + (qb * NQ + t) * L::kTileBytes;
                if (nkt > 0) ok = wait_all(bar(L::kQFull + qb), static_cast<uint32_t>(n / QB) & 1u);
                for (int j = 0; j < nkt && ok; ++j) {
                    const int s = (g + j) % S;
                    const uint32_t u = static_cast<uint32_t>((g + j) / S);
                    ok = wait_all(bar(L::kKFull + s), u & 1u);
                    // S overwrites the tile's S buffer once the softmax has read the previous one
                    if (ok && cs >= 1) ok = wait_all(bar(L::kSEmpty + t), static_cast<uint32_t>(cs - 1) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t k_sm = sb + L::kK + s * L::kTileBytes;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                            mma_bf16_ss(s_acc, sdesc_sw128(q_sm + koff, 16, 1024), sdesc_sw128(k_sm + koff, 16, 1024),
                                        kIdS, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(L::kSFull + t));
                        if (j == nkt - 1) mma_commit(bar(L::kQEmpty + qb));  // last read of this Q tile
                    }
                    __syncwarp();
                    issued = true;
                    ++cs;
                    if (j >= 1) issue_pv(j - 1, cs - 2);
                }
                if (ok && nkt > 0) issue_pv(nkt - 1, cs - 1);
                if (!ok) break;
                // Tiles and Q buffers this tile does not read are released in
                // order behind its earlier products (a commit arrives only once
                // everything this thread issued before it has completed).
                if (elect_one()) {
                    if (nkt == 0) mma_commit(bar(L::kQEmpty + qb));
                    for (int j = nkt; j < n_kt; ++j) mma_commit(bar(L::kKVEmpty + t * S + (g + j) % S));
                }
                __syncwarp();
                g += n_kt;
                if (nkt > 0) ++e;
            }
            // Drain: every MMA this warp issued has completed before TMEM is freed.
            if (issued) {
                if (elect_one()) mma_commit(bar(L::kDrain + t));
                __syncwarp();
                mbar_wait(bar(L::kDrain + t), 0, p.status);
            }
        }
    } else {
        if (NQ == 2) regs_inc<L::kRegsSoftmax>();
        // ---------------------------------------------------------- softmax
        const int t = warp >> 2;               // query tile of this warpgroup
        const int row = threadIdx.x & 127;     // == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_off + L::kSCol + t * 128;
        const uint32_t o_tm = tmem + lane_off + L::kOCol + t * D;
        const uint32_t p_tm = tmem + lane_off + L::kPCol + t * 64;
        const uint32_t plo_tm = tmem + lane_off + L::kPLoCol + t * 64;
        const uint32_t plo_sm = sb + L::kPLo + t * L::kPBytes;
        const float sl2 = p.scale_log2;
        // waits return the same verdict to every lane (tcgen05.ld/st below
        // are warp-collective)
        auto wait_w = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, p.status));
        };
        bool ok = true;
        int cs = 0;  // S products of this tile consumed so far, all items
        int ne = 0;  // epilogues this warpgroup has finished
        // The staging buffer may be rewritten once the previous epilogue's TMA
        // store has read it: its issuing thread (row 0) checks and signals.
        auto stage_free = [&]() {
            if (row == 0) {
                bulk_wait_read0();
                mbar_arrive(bar(L::kStageFree + t));
            }
            return wait_w(bar(L::kStageFree + t), static_cast<uint32_t>(ne - 1) & 1u);
        };
        if (L::kTmaStoreO && t == 0 && threadIdx.x == 0) tma_prefetch_desc(&tm_o);
        for (int r = 0; ok; ++r) {
            const int it = fwd_item(r);
            if (it >= p.n_items) break;
            const int bh = item_bh(it), cq = item_cq(it);
            const int nkt = tile_nkt(it, t);
            if (nkt == 0) continue;
            const int q0 = tile_q0(cq, t);
            const int qrow = q0 + row;
            float M = -INFINITY;  // running max of raw scores
            int C = 0;            // running count of keys equal to M (only C > 1 kept outside statistics)
            bool tied = false;    // statistics variant: C > 1 as the timed variant decides it
            float m = -INFINITY;  // current shift, raw units
            float mc = -INFINITY; // m * sl2
            float l = 0.f;
            int ones0 = 0, ones1 = 0;
            // mode 1 with a tolerance: the row's shift, found by a pre-pass
            // over the whole row, holds from the first key tile on
            const float m_fix = (MODE == 1 && p.shift && qrow < p.N) ? p.shift[static_cast<size_t>(bh) * p.N + qrow] : 0.f;
            for (int j = 0; j < nkt; ++j, ++cs) {
                ok = wait_w(bar(L::kSFull + t), static_cast<uint32_t>(cs) & 1u);
                if (!ok) break;
                tc_fence_after();
                float s[kBlockN];
                {
                    uint32_t rr[kBlockN / 32][32];
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c) tmem_ld32(s_tm + c * 32, rr[c]);
                    tmem_wait_ld();  // one wait for all four loads
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(rr[c][e]);
                }
                tc_fence_before();
                mbar_arrive(bar(L::kSEmpty + t));  // S is in registers: the next S may land

                const int k0 = j * kBlockN;
                const bool need_mask = CAUSAL ? (k0 + kBlockN > q0) : (k0 + kBlockN > p.N);
                if (need_mask) {
                    const int lim = CAUSAL ? (qrow - k0) : (p.N - 1 - k0);  // keep keys c <= lim
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        if (c > lim) s[c] = -INFINITY;
                }
                // row max: 3-input max instructions in 8 independent chains;
                // chain e holds the maximum of the keys c = e (mod 8)
                float tm;
                float mx[8];
                {
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = fmaxf(s[e], s[8 + e]);
#pragma unroll
                    for (int c = 16; c < kBlockN; c += 16)
#pragma unroll
                        for (int e = 0; e < 8; ++e) mx[e] = fmax3(mx[e], s[c + e], s[c + 8 + e]);
                    tm = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                }
                if (MODE == 1 && !STATS) {
                    // Only C > 1 matters here.  A tile max equal to the running
                    // max adds at least one tie to the C >= 1 already counted, so
                    // C > 1 follows without a count; only a new running max needs
                    // to know whether the tile holds it twice.
                    const bool newmax = tm > M;
                    const bool same = tm == M;
                    if (__any_sync(0xffffffffu, newmax)) {
                        const bool rep2 = tile_max_repeats(s, mx, tm);
                        if (newmax) {
                            M = tm;
                            C = rep2 ? 2 : 1;
                        }
                    }
                    if (same) C = 2;
                } else if (STATS) {
                    // Exact running tie count (reported per row).  The tile's count
                    // matters only where the tile max reaches the running max; warps
                    // where no row does skip it.
                    int tc = 0;
                    if (__any_sync(0xffffffffu, tm >= M)) {
                        int tcs[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
                        for (int c = 0; c < kBlockN; c += 8)
#pragma unroll
                            for (int e = 0; e < 8; ++e) tcs[e] += (s[c + e] == tm) ? 1 : 0;
                        tc = ((tcs[0] + tcs[1]) + (tcs[2] + tcs[3])) + ((tcs[4] + tcs[5]) + (tcs[6] + tcs[7]));
                    }
                    // the shift follows the same decision as in the timed
                    // variant (tile_max_repeats), so that the unit-probability
                    // counts reported here check it against the exact count
                    if (tm > M) {
                        M = tm;
                        C = tc;
                        tied = tile_max_repeats(s, mx, tm);
                    } else if (tm == M) {
                        tied = true;
                        C += tc;
                    }
                } else {
                    M = fmaxf(M, tm);
                }
                float m_new = M;
                if (MODE == 1 && p.shift) {
                    m_new = m_fix;
                } else if (MODE == 1 && (STATS ? tied : C > 1)) {
                    if (M > 0.f) m_new = p.beta * M;
                    else if (M < 0.f) m_new = 0.f;
                }
                const float mc_new = m_new * sl2;
                const bool changed = (m_new != m);
                const float rsc = changed ? ex2_approx(mc - mc_new) : 1.f;
                m = m_new;
                mc = mc_new;
                // Pbar = exp2(s * alpha*log2e - m * alpha*log2e) with paired FP32 FMAs
                // and adds, packed to BF16 pairs in registers (plus the lo part in
                // mode 2).  This overlaps the previous tile's Pbar V on the tensor
                // core; only the stores below wait for it.
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                const uint64_t nmc2 = f2_pack(-mc_new, -mc_new);
                uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};  // 8 partial row sums, as 4 pairs
                int cnt = 0;
                uint32_t w[kBlockN / 2], wl[kBlockN / 2];  // wl unused (and eliminated) unless MODE == 2
#pragma unroll
                for (int e = 0; e < kBlockN / 2; ++e) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(s[2 * e], s[2 * e + 1]), sl2x2, nmc2), x0, x1);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    ls2[e & 3] = f2_add(ls2[e & 3], f2_pack(p0, p1));
                    w[e] = pack_bf16x2(p0, p1);
                    if (MODE == 2) {
                        // p - bf16(p) is exact in FP32; hi + lo carries ~16 bits of p
                        const float h0 = __uint_as_float(w[e] << 16);
                        const float h1 = __uint_as_float(w[e] & 0xFFFF0000u);
                        wl[e] = pack_bf16x2(p0 - h0, p1 - h1);
                    }
                    if (STATS) cnt += ((w[e] & 0xFFFFu) == 0x3F80u ? 1 : 0) + ((w[e] >> 16) == 0x3F80u ? 1 : 0);
                }
                // Pbar may overwrite the TMEM Pbar buffer and O may be rescaled
                // only after the previous Pbar V product (of this or the
                // previous item) has completed.
                if (cs >= 1) {
                    ok = wait_w(bar(L::kODone + t), static_cast<uint32_t>(cs - 1) & 1u);
                    if (!ok) break;
                }
                // FP32 output: the lo buffer held the previous item's O for its TMA store
                if (L::kTmaStoreO && !STATS && L::kLoInSmem && j == 0 && ne >= 1) {
                    ok = stage_free();
                    if (!ok) break;
                }
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    tmem_st16(p_tm + 16 * h, *reinterpret_cast<const uint32_t(*)[16]>(&w[16 * h]));
                    if (L::kLoInTmem) tmem_st16(plo_tm + 16 * h, *reinterpret_cast<const uint32_t(*)[16]>(&wl[16 * h]));
                    if (L::kLoInSmem) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int ch = (h & 1) * 4 + q;  // 16-byte chunk within the 128-byte row
                            st_shared_v4(plo_sm + (h >> 1) * 16384 + sw128_off(row, ch), wl[16 * h + 4 * q],
                                         wl[16 * h + 4 * q + 1], wl[16 * h + 4 * q + 2], wl[16 * h + 4 * q + 3]);
                        }
                    }
                }
                float lsum;
                {
                    float a0, a1;
                    f2_unpack(f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3])), a0, a1);
                    lsum = a0 + a1;
                }
                l = l * rsc + lsum;
                if (STATS) {
                    if (changed) ones1 = 0;
                    ones0 += cnt;
                    ones1 += cnt;
                }
                // rescale O after the scores are consumed (keeps register use low)
                if (j >= 1 && __any_sync(0xffffffffu, changed)) {
                    tc_fence_after();
                    uint32_t r[D / 32][32];
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tm + c * 32, r[c]);
                    tmem_wait_ld();  // one wait for all loads
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[c][e] = __float_as_uint(__uint_as_float(r[c][e]) * rsc);
                        tmem_st32(o_tm + c * 32, r[c]);
                    }
                }
                tmem_wait_st();  // Pbar (and any rescaled O) written to TMEM
                if (L::kLoInSmem) fence_async_smem();
                tc_fence_before();
                mbar_arrive(bar(L::kPFull + t));
            }
            if (!ok) break;
            // ------------------------------------------------------ epilogue
            // Read O out of TMEM (which frees it for the next item's first
            // product), then normalise and store O and the LSE.
            ok = wait_w(bar(L::kODone + t), static_cast<uint32_t>(cs - 1) & 1u);
            if (!ok) break;
            tc_fence_after();
            const bool store = qrow < p.N;
            const size_t rowid = static_cast<size_t>(bh) * p.N + qrow;
            if (STATS) {
                tc_fence_before();
                mbar_arrive(bar(L::kOFree + t));
                if (store) {
                    p.tie_count[rowid] = p.rs_in ? p.rs_in[rowid] : C;
                    if (p.p_one) {
                        p.p_one[rowid] = ones0;
                        p.p_one[static_cast<size_t>(p.BH) * p.N + rowid] = ones1;
                    }
                }
            } else {
                // tcgen05.ld is warp-collective: every lane loads, only rows < N store.
                uint32_t ov[D];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[c * 32]));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::kOFree + t));
                const float inv_l = 1.f / l;
                if (L::kTmaStoreO) {
                    // Rows go to the 128-byte-swizzled staging tile (the TMA
                    // box layout); rows past N are clipped by the TMA store.
                    const uint32_t stg = MODE == 2 ? plo_sm : sb + L::kOStage + t * L::kOStageBytes;
                    if (MODE != 2 && ne >= 1) {
                        ok = stage_free();
                        if (!ok) break;
                    }
                    if (MODE == 2) {
#pragma unroll
                        for (int c = 0; c < D / 4; ++c)  // 16-byte chunks of 4 floats; 32 columns per box
                            st_shared_v4(stg + (c >> 3) * 16384 + sw128_off(row, c & 7),
                                         __float_as_uint(__uint_as_float(ov[4 * c]) * inv_l),
                                         __float_as_uint(__uint_as_float(ov[4 * c + 1]) * inv_l),
                                         __float_as_uint(__uint_as_float(ov[4 * c + 2]) * inv_l),
                                         __float_as_uint(__uint_as_float(ov[4 * c + 3]) * inv_l));
                    } else {
#pragma unroll
                        for (int c = 0; c < D / 8; ++c)  // 16-byte chunks of 8 BF16
                            st_shared_v4(stg + sw128_off(row, c),
                                         pack_bf16x2(__uint_as_float(ov[8 * c + 0]) * inv_l, __uint_as_float(ov[8 * c + 1]) * inv_l),
                                         pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv_l, __uint_as_float(ov[8 * c + 3]) * inv_l),
                                         pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv_l, __uint_as_float(ov[8 * c + 5]) * inv_l),
                                         pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv_l, __uint_as_float(ov[8 * c + 7]) * inv_l));
                    }
                    fence_async_smem();
                    mbar_arrive(bar(L::kOStaged + t));
                    if (row == 0) {
                        ok = mbar_wait(bar(L::kOStaged + t), static_cast<uint32_t>(ne) & 1u, p.status);
                        if (ok) {
                            const int hh = bh % p.H, bb = bh / p.H;  // head and batch of the tile coordinates
                            if (MODE == 2) {
                                tma_store_rows(&tm_o, stg, 0, q0, hh, bb, p.lay.head_inner);
                                tma_store_rows(&tm_o, stg + 16384, 32, q0, hh, bb, p.lay.head_inner);
                            } else {
                                tma_store_rows(&tm_o, stg, 0, q0, hh, bb, p.lay.head_inner);
                            }
                            bulk_commit();
                        }
                    }
                } else if (store) {
                    if (MODE == 2) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + p.lay.row(bh, qrow));
#pragma unroll
                        for (int e = 0; e < D / 4; ++e)
                            dst[e] = make_float4(__uint_as_float(ov[4 * e]) * inv_l, __uint_as_float(ov[4 * e + 1]) * inv_l,
                                                 __uint_as_float(ov[4 * e + 2]) * inv_l,
                                                 __uint_as_float(ov[4 * e + 3]) * inv_l);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + p.lay.row(bh, qrow));
#pragma unroll
                        for (int e = 0; e < D / 8; ++e) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv_l, __uint_as_float(ov[8 * e + 1]) * inv_l);
                            w.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv_l, __uint_as_float(ov[8 * e + 3]) * inv_l);
                            w.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv_l, __uint_as_float(ov[8 * e + 5]) * inv_l);
                            w.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv_l, __uint_as_float(ov[8 * e + 7]) * inv_l);
                            dst[e] = w;
                        }
                    }
                }
                // LSE = m*alpha + ln(l), natural log of the scaled-score normaliser
                if (store) {
                    const float lse = (mc + lg2_approx(l)) * 0.69314718055994531f;
                    p.lse[rowid] = lse;
                    // l = 0 (every Pbar underflowed) or a NaN from 0 * inf in
                    // a rescale: reported through the status word
                    if (!isfinite(lse)) atomicOr(p.status, kDevNonFinite);
                }
            }
            ++ne;
        }
    }

    // O's TMA stores complete before the CTA exits
    if (L::kTmaStoreO && !STATS && warp < kProducerWarp && (threadIdx.x & 127) == 0) bulk_wait0();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// Two query tiles per CTA where shared memory allows it (d = 64).
template <int D>
constexpr int kQTilesPerCta = (D == 64) ? 2 : 1;

template <int D, int MODE, bool CAUSAL, bool STATS>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
    constexpr int NQ = kQTilesPerCta<D>;
    using L = FwdLayout<D, MODE, NQ>;
    auto kern = fwd_kernel<D, MODE, CAUSAL, STATS, NQ>;
    static unsigned smem_set = 0;  // devices on which this instantiation's limit is raised
    cudaError_t e = smem_limit_once(kern, L::kAlloc, &smem_set);
    if (e != cudaSuccess) {
        set_error("fwd cudaFuncSetAttribute", e);
        return e;
    }
    FwdParams p;
    p.o = a.o;
    p.lse = a.lse;
    p.tie_count = a.tie_count;
    p.p_one = a.p_one;
    p.BH = a.BH;
    p.N = a.N;
    p.scale_log2 = a.scale_log2;
    p.beta = a.beta;
    p.status = a.status;
    p.test_withhold_k = a.test_withhold_k;
    p.shift = a.shift;
    p.rs_in = a.rs_in;
    p.H = a.lay.H;
    p.lay = a.lay;
    // ~0: every head (H may exceed 64); else a set of heads h < H <= 64
    const uint64_t all = p.H >= 64 ? ~0ull : ((1ull << p.H) - 1ull);
    p.head_mask = a.head_mask & all;
    p.Hon = (a.head_mask == ~0ull) ? p.H : __builtin_popcountll(p.head_mask);
    p.BHon = a.BH / p.H * p.Hon;
    const int n_qt = (a.N + kBlockM - 1) / kBlockM;
    p.n_cq = (n_qt + NQ - 1) / NQ;
    p.n_items = p.BHon * p.n_cq;
    // persistent: one CTA per SM (or per item, if fewer)
    const int n_cta = p.n_items < a.num_sms ? p.n_items : a.num_sms;
    dim3 grid(static_cast<unsigned>(n_cta > 0 ? n_cta : 1));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // set-up overlaps the previous kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_begin(STATS ? 1 : 0, stream);
    e = cudaLaunchKernelEx(&cfg, kern, *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o, p);
    prof_end(STATS ? 1 : 0, stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) set_error("fwd launch", e);
    return e;
}

template <int D, int MODE>
cudaError_t dispatch_causal(const FwdArgs& a, bool stats, cudaStream_t st) {
    if (a.causal) return stats ? launch_fwd_t<D, MODE, true, true>(a, st) : launch_fwd_t<D, MODE, true, false>(a, st);
    return stats ? launch_fwd_t<D, MODE, false, true>(a, st) : launch_fwd_t<D, MODE, false, false>(a, st);
}

template <int D>
cudaError_t dispatch_mode(const FwdArgs& a, bool stats, cudaStream_t st) {
    switch (a.mode) {
        case 0: return dispatch_causal<D, 0>(a, stats, st);
        case 1: return dispatch_causal<D, 1>(a, stats, st);
        default: return dispatch_causal<D, 2>(a, stats, st);
    }
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, bool stats, cudaStream_t stream) {
    return a.d == 64 ? dispatch_mode<64>(a, stats, stream) : dispatch_mode<128>(a, stats, stream);
}

}  // namespace fa
