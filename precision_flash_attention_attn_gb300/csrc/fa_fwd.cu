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
//   warp 4*NQ+1  MMA issuer: S_t = Q_t K_j^T into tile t's TMEM S buffer,
//              then O_t += Pbar_t V_j (tcgen05.mma kind::f16; Q, K, V from
//              shared memory, Pbar from tensor memory).  With two query tiles the two softmax
//              warpgroups overlap each other's MMAs and share every K/V tile.
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
    static constexpr int kStages = (D == 64) ? (kLoInSmem ? 3 : 4) : 3;
    static constexpr int kQ = 0;                                  // [NQ]
    static constexpr int kK = kQ + NQ * kTileBytes;               // [kStages]
    static constexpr int kV = kK + kStages * kTileBytes;          // [kStages]
    static constexpr int kPLo = kV + kStages * kTileBytes;        // [NQ], mode 2 without TMEM room
    static constexpr int kBar = kPLo + (kLoInSmem ? NQ * kPBytes : 0);
    // barriers
    static constexpr int kQFull = 0;
    static constexpr int kKFull = 1;
    static constexpr int kVFull = kKFull + kStages;
    static constexpr int kKVEmpty = kVFull + kStages;
    static constexpr int kSFull = kKVEmpty + kStages;  // [NQ]
    static constexpr int kSEmpty = kSFull + NQ;        // [NQ]
    static constexpr int kPFull = kSEmpty + NQ;        // [NQ]
    static constexpr int kODone = kPFull + NQ;         // [NQ]
    static constexpr int kDrain = kODone + NQ;
    static constexpr int kNumBars = kDrain + 1;
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
    static constexpr int kThreads = 128 * NQ + 64;
    static_assert(kAlloc <= 232448, "shared memory budget");
};

struct FwdParams {
    void* o;
    float* lse;
    int32_t* tie_count;
    int32_t* p_one;
    int BH, N;
    float scale_log2;
    int* status;
};

template <int D, int MODE, bool CAUSAL, bool STATS, int NQ>
__global__ void __launch_bounds__(128 * NQ + 64, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using L = FwdLayout<D, MODE, NQ>;
    constexpr int S = L::kStages;
    constexpr int kProducerWarp = 4 * NQ;
    constexpr int kMmaWarp = 4 * NQ + 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + L::kBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int cq = gridDim.y - 1 - blockIdx.y;  // longest causal tiles first
    const int n_ktiles_all = (p.N + kBlockN - 1) / kBlockN;
    // per query tile: first row and number of key tiles it visits (0: past N)
    int q0s[NQ], nkts[NQ];
    int n_kt = 0, n_active = 0;
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
        const int qt = cq * NQ + t;
        q0s[t] = qt * kBlockM;
        const bool active = q0s[t] < p.N;
        nkts[t] = !active ? 0 : (CAUSAL ? (qt + 1 < n_ktiles_all ? qt + 1 : n_ktiles_all) : n_ktiles_all);
        n_kt = nkts[t] > n_kt ? nkts[t] : n_kt;
        n_active += active ? 1 : 0;
    }

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kQFull), 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(L::kKFull + s), 1);
            mbar_init(bar(L::kVFull + s), 1);
            mbar_init(bar(L::kKVEmpty + s), 1);
        }
        for (int t = 0; t < NQ; ++t) {
            mbar_init(bar(L::kSFull + t), 1);
            mbar_init(bar(L::kSEmpty + t), 128);
            mbar_init(bar(L::kPFull + t), 128);
            mbar_init(bar(L::kODone + t), 1);
        }
        mbar_init(bar(L::kDrain), 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sb + L::kTmemSlot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(bar(L::kQFull), L::kTileBytes * n_active);
            for (int t = 0; t < NQ; ++t) {
                if (nkts[t] == 0) continue;
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sb + L::kQ + t * L::kTileBytes + b * 16384, &tm_q, bar(L::kQFull), b * 64, q0s[t],
                                bh);
            }
            int issued = 0;
            for (int j = 0; j < n_kt; ++j) {
                const int s = j % S;
                const uint32_t u = static_cast<uint32_t>(j / S);
                if (j >= S && !mbar_wait(bar(L::kKVEmpty + s), (u - 1) & 1u, p.status)) break;
                mbar_arrive_expect_tx(bar(L::kKFull + s), L::kTileBytes);
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sb + L::kK + s * L::kTileBytes + b * 16384, &tm_k, bar(L::kKFull + s),
                                b * 64, j * kBlockN, bh);
                mbar_arrive_expect_tx(bar(L::kVFull + s), L::kTileBytes);
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(sb + L::kV + s * L::kTileBytes + b * 16384, &tm_v, bar(L::kVFull + s),
                                b * 64, j * kBlockN, bh);
                issued = j + 1;
            }
            // Every copy this thread issued must have landed before the CTA
            // may exit (normally long since true).
            mbar_wait(bar(L::kQFull), 0, p.status);
            for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j) {
                const uint32_t u = static_cast<uint32_t>(j / S);
                mbar_wait(bar(L::kKFull + j % S), u & 1u, p.status);
                mbar_wait(bar(L::kVFull + j % S), u & 1u, p.status);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16(kBlockM, kBlockN, false, false);
            constexpr uint32_t kIdPV = idesc_bf16(kBlockM, D, false, true);
            bool ok = mbar_wait(bar(L::kQFull), 0, p.status);
            auto issue_pv = [&](int jj) {
                const int s = jj % S;
                const uint32_t u = static_cast<uint32_t>(jj / S);
                ok = ok && mbar_wait(bar(L::kVFull + s), u & 1u, p.status);
#pragma unroll
                for (int t = 0; t < NQ; ++t) {
                    if (jj >= nkts[t]) continue;
                    ok = ok && mbar_wait(bar(L::kPFull + t), static_cast<uint32_t>(jj) & 1u, p.status);
                    if (!ok) return;
                    tc_fence_after();
                    const uint32_t o_t = tmem + L::kOCol + t * D;
                    // A = Pbar from TMEM: 16 keys (8 columns) per MMA step
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk) {
                        const uint64_t b = sdesc_sw128(sb + L::kV + s * L::kTileBytes + kk * 2048, 16384, 1024);
                        mma_bf16_ts(o_t, tmem + L::kPCol + t * 64 + kk * 8, b, kIdPV, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (L::kLoInTmem) {
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk) {
                            const uint64_t b = sdesc_sw128(sb + L::kV + s * L::kTileBytes + kk * 2048, 16384, 1024);
                            mma_bf16_ts(o_t, tmem + L::kPLoCol + t * 64 + kk * 8, b, kIdPV, 1u);
                        }
                    } else if (L::kLoInSmem) {
#pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk) {
                            const uint64_t a = sdesc_sw128(
                                sb + L::kPLo + t * L::kPBytes + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                            const uint64_t b = sdesc_sw128(sb + L::kV + s * L::kTileBytes + kk * 2048, 16384, 1024);
                            mma_bf16_ss(o_t, a, b, kIdPV, 1u);
                        }
                    }
                    mma_commit(bar(L::kODone + t));
                }
                if (ok) mma_commit(bar(L::kKVEmpty + s));
            };
            for (int j = 0; j < n_kt && ok; ++j) {
                const int s = j % S;
                const uint32_t u = static_cast<uint32_t>(j / S);
                ok = mbar_wait(bar(L::kKFull + s), u & 1u, p.status);
#pragma unroll
                for (int t = 0; t < NQ; ++t) {
                    if (!ok || j >= nkts[t]) continue;
                    if (j >= 1)
                        ok = mbar_wait(bar(L::kSEmpty + t), static_cast<uint32_t>(j - 1) & 1u, p.status);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint64_t a = sdesc_sw128(sb + L::kQ + t * L::kTileBytes + koff, 16, 1024);
                        const uint64_t b = sdesc_sw128(sb + L::kK + s * L::kTileBytes + koff, 16, 1024);
                        mma_bf16_ss(tmem + L::kSCol + t * 128, a, b, kIdS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(L::kSFull + t));
                }
                if (ok && j >= 1) issue_pv(j - 1);
            }
            if (ok && n_kt > 0) issue_pv(n_kt - 1);
            // Drain: every MMA issued above has completed before TMEM is freed.
            mma_commit(bar(L::kDrain));
            mbar_wait(bar(L::kDrain), 0, p.status);
        }
    } else {
        // ---------------------------------------------------------- softmax
        const int t = warp >> 2;               // query tile of this warpgroup
        const int row = threadIdx.x & 127;     // == TMEM lane
        const int q0 = q0s[t];
        const int nkt = nkts[t];
        const int qrow = q0 + row;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_off + L::kSCol + t * 128;
        const uint32_t o_tm = tmem + lane_off + L::kOCol + t * D;
        const uint32_t p_tm = tmem + lane_off + L::kPCol + t * 64;
        const uint32_t plo_tm = tmem + lane_off + L::kPLoCol + t * 64;
        const uint32_t plo_sm = sb + L::kPLo + t * L::kPBytes;
        const float sl2 = p.scale_log2;
        float M = -INFINITY;  // running max of raw scores
        int C = 0;            // running count of keys equal to M
        float m = -INFINITY;  // current shift, raw units
        float mc = -INFINITY; // m * sl2
        float l = 0.f;
        int ones0 = 0, ones1 = 0;
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            ok = mbar_wait(bar(L::kSFull + t), static_cast<uint32_t>(j) & 1u, p.status);
            if (!ok) break;
            tc_fence_after();
            float s[kBlockN];
            {
                uint32_t r[kBlockN / 32][32];
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c) tmem_ld32(s_tm + c * 32, r[c]);
                tmem_wait_ld();  // one wait for all four loads
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[c][e]);
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
            // row max: 3-input max instructions in 8 independent chains
            float tm;
            {
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx[e] = fmaxf(s[e], s[8 + e]);
#pragma unroll
                for (int c = 16; c < kBlockN; c += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = fmax3(mx[e], s[c + e], s[c + 8 + e]);
                tm = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            }
            if (MODE == 1 || STATS) {
                // The tile's tie count matters only where the tile max reaches
                // the running max; warps where no row does skip the count (the
                // common case once the max has settled).
                int tc = 0;
                if (__any_sync(0xffffffffu, tm >= M)) {
                    int tcs[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
                    for (int c = 0; c < kBlockN; c += 8)
#pragma unroll
                        for (int e = 0; e < 8; ++e) tcs[e] += (s[c + e] == tm) ? 1 : 0;
                    tc = ((tcs[0] + tcs[1]) + (tcs[2] + tcs[3])) + ((tcs[4] + tcs[5]) + (tcs[6] + tcs[7]));
                }
                if (tm > M) {
                    M = tm;
                    C = tc;
                } else if (tm == M) {
                    C += tc;
                }
            } else {
                M = fmaxf(M, tm);
            }
            float m_new = M;
            if (MODE == 1 && C > 1) {
                if (M > 0.f) m_new = kStabBeta * M;
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
            // Pbar_j may overwrite the TMEM Pbar buffer and O may be rescaled
            // only after O += Pbar_{j-1} V_{j-1} has completed.
            if (j >= 1) {
                ok = mbar_wait(bar(L::kODone + t), static_cast<uint32_t>(j - 1) & 1u, p.status);
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
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(o_tm + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * rsc);
                    tmem_st32(o_tm + c * 32, r);
                }
            }
            tmem_wait_st();  // Pbar (and any rescaled O) written to TMEM
            if (L::kLoInSmem) fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar(L::kPFull + t));
        }
        if (ok && nkt > 0) ok = mbar_wait(bar(L::kODone + t), static_cast<uint32_t>(nkt - 1) & 1u, p.status);
        const bool store = ok && nkt > 0 && qrow < p.N;
        const size_t rowid = static_cast<size_t>(bh) * p.N + qrow;
        if (STATS) {
            if (store) {
                p.tie_count[rowid] = C;
                if (p.p_one) {
                    p.p_one[rowid] = ones0;
                    p.p_one[static_cast<size_t>(p.BH) * p.N + rowid] = ones1;
                }
            }
        } else if (nkt > 0 && __all_sync(0xffffffffu, ok)) {
            // tcgen05.ld is warp-collective: every lane loads, only rows < N store.
            tc_fence_after();
            const float inv_l = 1.f / l;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(o_tm + c * 32, r);
                tmem_wait_ld();
                if (!store) continue;
                if (MODE == 2) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + rowid * D + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv_l, __uint_as_float(r[4 * e + 1]) * inv_l,
                                             __uint_as_float(r[4 * e + 2]) * inv_l, __uint_as_float(r[4 * e + 3]) * inv_l);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + rowid * D + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * inv_l, __uint_as_float(r[8 * e + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * inv_l, __uint_as_float(r[8 * e + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * inv_l, __uint_as_float(r[8 * e + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * inv_l, __uint_as_float(r[8 * e + 7]) * inv_l);
                        dst[e] = w;
                    }
                }
            }
            // LSE = m*alpha + ln(l), natural log of the scaled-score normaliser
            if (store) p.lse[rowid] = (mc + lg2_approx(l)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
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
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
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
    p.status = a.status;
    const int n_qt = (a.N + kBlockM - 1) / kBlockM;
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>((n_qt + NQ - 1) / NQ));
    prof_begin(STATS ? 1 : 0, stream);
    kern<<<grid, L::kThreads, L::kAlloc, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
    prof_end(STATS ? 1 : 0, stream);
    e = cudaGetLastError();
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
