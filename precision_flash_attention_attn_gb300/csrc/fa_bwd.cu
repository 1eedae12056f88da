// Flash-attention backward for sm_103a, recomputing P from the saved LSE.
//
// For loss gradient dO and stored output O of the same mode ("Why
// Low-Precision Transformer Training Fails: An Analysis on Flash Attention",
// sections 3.4.2-3.4.3):
//   delta = rowsum(dO o O)                (O as stored: BF16, or FP32 in mode 2)
//   P     = exp(alpha * Q K^T - LSE)
//   dP    = dO V^T
//   dS    = alpha * P o (dP - delta)
//   dQ    = dS K,   dK = dS^T Q,   dV = P^T dO   (dK, dV: textbook gradients)
//
// Kernels, in stream order:
//   bwd_pre_kernel   -LSE*log2(e) and -alpha*delta per row into padded
//                    workspaces, zero the FP32 dQ accumulator.
//   bwd_kernel       one CTA per (batch*head, 128-key tile); K and V stay in
//                    shared memory while the CTA walks the 128-query tiles
//                    (causal: only tiles at or below the diagonal).  Per query
//                    tile, five tcgen05 MMAs:
//                      S^T  = K Q^T      (TMEM, FP32)
//                      dP^T = V dO^T     (TMEM, FP32)
//                      dV  += P^T dO     (TMEM accumulator)
//                      dK  += dS^T Q     (TMEM accumulator)
//                      dQ_t = dS K       (TMEM), added to the FP32 workspace
//                                        with TMA reduce-add
//                    Warp roles: two math warpgroups (warps 0-3: query
//                    columns 0-63 of the tile, warps 4-7: columns 64-127;
//                    thread t of a warpgroup owns key row t) recompute P^T and
//                    dS^T, drain each dQ tile from TMEM into the reduce-add
//                    (one 32-row box per warp), and finally store dK and dV;
//                    warp 8 issues TMA loads; warp 9 issues the MMAs.  The
//                    next tile's S^T and dP^T are issued ahead of the current
//                    tile's dK/dQ products.
//   dq_convert_kernel  dQ workspace (FP32) -> BF16.
#include <cuda_bf16.h>

#include <cstdio>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

// ------------------------------------------------------------- preprocess --

// D/8 threads per row, 8 elements (16 bytes of dO) each; rows padded to Npad.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
    constexpr int TPR = D / 8;       // threads per row
    constexpr int RPW = 32 / TPR;    // rows per warp and pass
    const int lane = threadIdx.x & 31;
    const int sub = lane % TPR;
    const long long rows = static_cast<long long>(a.BH) * a.Npad;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long gw = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const float log2e = 1.4426950408889634f;
    for (long long r0 = gw * RPW; r0 < rows; r0 += nwarps * RPW) {
        const long long r = r0 + lane / TPR;
        const int bh = static_cast<int>(r / a.Npad);
        const int i = static_cast<int>(r % a.Npad);
        const bool valid = r < rows && i < a.N;
        float acc = 0.f;
        if (valid) {
            const size_t base = (static_cast<size_t>(bh) * a.N + i) * D + sub * 8;
            const uint4 g = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + base);
            const uint32_t gw4[4] = {g.x, g.y, g.z, g.w};
            if (a.mode == 2) {
                const float4 o0 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.o) + base);
                const float4 o1 = *reinterpret_cast<const float4*>(static_cast<const float*>(a.o) + base + 4);
                const float of[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(__uint_as_float(gw4[e] << 16), of[2 * e], acc);
                    acc = fmaf(__uint_as_float(gw4[e] & 0xFFFF0000u), of[2 * e + 1], acc);
                }
            } else {
                const uint4 o = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.o) + base);
                const uint32_t ow4[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(__uint_as_float(gw4[e] << 16), __uint_as_float(ow4[e] << 16), acc);
                    acc = fmaf(__uint_as_float(gw4[e] & 0xFFFF0000u), __uint_as_float(ow4[e] & 0xFFFF0000u), acc);
                }
            }
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (sub == 0 && r < rows) {
            // stored pre-negated / pre-scaled for the main kernel's FMAs:
            //   P  = exp2(s * alpha*log2e + lse2),  lse2 = -LSE*log2e
            //   dS = P * (alpha * dP + delta),      delta = -alpha * rowsum(dO o O)
            a.delta[r] = valid ? -a.scale * acc : 0.f;
            // padded rows: P = exp2(s - inf) = 0
            a.lse2[r] = valid ? -a.lse[static_cast<size_t>(bh) * a.N + i] * log2e : -INFINITY;
        }
    }
    // zero the dQ accumulator
    const size_t n4 = static_cast<size_t>(a.BH) * a.N * D / 4;
    float4* acc4 = reinterpret_cast<float4*>(a.dq_acc);
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n4; e += stride)
        acc4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                         size_t n8) {
    for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n8;
         e += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 x = reinterpret_cast<const float4*>(acc)[2 * e];
        const float4 y = reinterpret_cast<const float4*>(acc)[2 * e + 1];
        uint4 w;
        w.x = pack_bf16x2(x.x, x.y);
        w.y = pack_bf16x2(x.z, x.w);
        w.z = pack_bf16x2(y.x, y.y);
        w.w = pack_bf16x2(y.z, y.w);
        reinterpret_cast<uint4*>(dq)[e] = w;
    }
}

// ---------------------------------------------------------------- main ----

template <int D>
struct BwdLayout {
    static constexpr int kTile = kBlockM * D * 2;      // 128 rows x D BF16
    static constexpr int kQStages = (D == 64) ? 2 : 1;
    static constexpr int kK = 0;
    static constexpr int kV = kK + kTile;
    static constexpr int kQ = kV + kTile;                       // [kQStages]
    static constexpr int kDO = kQ + kQStages * kTile;           // [kQStages]
    static constexpr int kPt = kDO + kQStages * kTile;          // 128 keys x 128 queries BF16
    static constexpr int kDSt = kPt + kBlockM * kBlockN * 2;
    static constexpr int kStage = kDSt + kBlockM * kBlockN * 2; // 8 warps x (32 x 32 FP32), swizzled
    static constexpr int kLse = kStage + 8 * 4096;              // [kQStages][128] FP32 (-LSE*log2e)
    static constexpr int kDelta = kLse + kQStages * 512;        // [kQStages][128] FP32 (-alpha*delta)
    static constexpr int kBar = kDelta + kQStages * 512;
    // barriers
    static constexpr int kKVFull = 0;
    static constexpr int kQFull = 1;                       // [kQStages]
    static constexpr int kQEmpty = kQFull + kQStages;      // [kQStages]
    static constexpr int kSFull = kQEmpty + kQStages;
    static constexpr int kSEmpty = kSFull + 1;
    static constexpr int kDPFull = kSEmpty + 1;
    static constexpr int kDPEmpty = kDPFull + 1;
    static constexpr int kPFull = kDPEmpty + 1;
    static constexpr int kDSFull = kPFull + 1;
    static constexpr int kPDSFree = kDSFull + 1;
    static constexpr int kDQFull = kPDSFree + 1;
    static constexpr int kDQEmpty = kDQFull + 1;
    static constexpr int kDKVDone = kDQEmpty + 1;
    static constexpr int kNumBars = kDKVDone + 1;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kBytes = kTmemSlot + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColDP = 128;
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
    static constexpr bool kDQAliasS = (D != 64);  // no room for a separate dQ tile at d = 128
    static constexpr uint32_t kColDQ = kDQAliasS ? kColS : 256 + 2 * D;
    static constexpr uint32_t kMathThreads = 256;  // two warpgroups
};

struct BwdParams {
    float* lse2;
    float* delta;
    void* dk;
    void* dv;
    int BH, N, Npad;
    float scale, scale_log2;
    int* status;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqacc, const BwdParams p) {
    using L = BwdLayout<D>;
    constexpr int QS = L::kQStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + L::kBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int kt = blockIdx.y;  // causal: key tile 0 has the most query tiles, runs first
    const int k0 = kt * kBlockN;
    const int n_qt_all = (p.N + kBlockM - 1) / kBlockM;
    const int qt_begin = CAUSAL ? kt : 0;
    const int n_iter = n_qt_all - qt_begin;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kKVFull), 1);
        for (int s = 0; s < QS; ++s) {
            mbar_init(bar(L::kQFull + s), 1);
            mbar_init(bar(L::kQEmpty + s), 1);
        }
        mbar_init(bar(L::kSFull), 1);
        mbar_init(bar(L::kSEmpty), L::kMathThreads);
        mbar_init(bar(L::kDPFull), 1);
        mbar_init(bar(L::kDPEmpty), L::kMathThreads);
        mbar_init(bar(L::kPFull), L::kMathThreads);
        mbar_init(bar(L::kDSFull), L::kMathThreads);
        mbar_init(bar(L::kPDSFree), 1);
        mbar_init(bar(L::kDQFull), 1);
        mbar_init(bar(L::kDQEmpty), L::kMathThreads);
        mbar_init(bar(L::kDKVDone), 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(sb + L::kTmemSlot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

    if (warp == 8) {
        // -------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            mbar_arrive_expect_tx(bar(L::kKVFull), 2 * L::kTile);
            for (int b = 0; b < D / 64; ++b) {
                tma_load_3d(sb + L::kK + b * 16384, &tm_k, bar(L::kKVFull), b * 64, k0, bh);
                tma_load_3d(sb + L::kV + b * 16384, &tm_v, bar(L::kKVFull), b * 64, k0, bh);
            }
            int issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it % QS;
                const uint32_t u = static_cast<uint32_t>(it / QS);
                if (it >= QS && !mbar_wait(bar(L::kQEmpty + s), (u - 1) & 1u, p.status)) break;
                const int q0 = (qt_begin + it) * kBlockM;
                mbar_arrive_expect_tx(bar(L::kQFull + s), 2 * L::kTile + 1024);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_3d(sb + L::kQ + s * L::kTile + b * 16384, &tm_q, bar(L::kQFull + s), b * 64, q0, bh);
                    tma_load_3d(sb + L::kDO + s * L::kTile + b * 16384, &tm_do, bar(L::kQFull + s), b * 64, q0, bh);
                }
                const size_t roff = static_cast<size_t>(bh) * p.Npad + q0;
                bulk_load(sb + L::kLse + s * 512, p.lse2 + roff, 512, bar(L::kQFull + s));
                bulk_load(sb + L::kDelta + s * 512, p.delta + roff, 512, bar(L::kQFull + s));
                issued = it + 1;
            }
            mbar_wait(bar(L::kKVFull), 0, p.status);
            for (int it = issued - QS > 0 ? issued - QS : 0; it < issued; ++it)
                mbar_wait(bar(L::kQFull + it % QS), static_cast<uint32_t>(it / QS) & 1u, p.status);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdSS = idesc_bf16(kBlockM, kBlockN, false, false);  // S^T, dP^T
            constexpr uint32_t kIdAcc = idesc_bf16(kBlockM, D, false, true);         // dV, dK
            constexpr uint32_t kIdDQ = idesc_bf16(kBlockM, D, true, true);           // dQ
            bool ok = mbar_wait(bar(L::kKVFull), 0, p.status);
            // S^T(it) = K Q^T
            auto issue_s = [&](int it) {
                const int s = it % QS;
                ok = ok && mbar_wait(bar(L::kQFull + s), static_cast<uint32_t>(it / QS) & 1u, p.status);
                if (ok && it >= 1) ok = mbar_wait(bar(L::kSEmpty), static_cast<uint32_t>(it - 1) & 1u, p.status);
                if (ok && it >= 1 && L::kDQAliasS)
                    ok = mbar_wait(bar(L::kDQEmpty), static_cast<uint32_t>(it - 1) & 1u, p.status);
                if (!ok) return;
                tc_fence_after();
                const uint32_t sQ = sb + L::kQ + s * L::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16_ss(tmem + L::kColS, sdesc_sw128(sb + L::kK + ko, 16, 1024), sdesc_sw128(sQ + ko, 16, 1024),
                                kIdSS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kSFull));
            };
            // dP^T(it) = V dO^T   (Q/dO stage it is already known to be loaded)
            auto issue_dp = [&](int it) {
                const int s = it % QS;
                if (ok && it >= 1) ok = mbar_wait(bar(L::kDPEmpty), static_cast<uint32_t>(it - 1) & 1u, p.status);
                if (!ok) return;
                tc_fence_after();
                const uint32_t sDO = sb + L::kDO + s * L::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16_ss(tmem + L::kColDP, sdesc_sw128(sb + L::kV + ko, 16, 1024), sdesc_sw128(sDO + ko, 16, 1024),
                                kIdSS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kDPFull));
            };
            // Software pipeline: the next tile's S^T (and dP^T) are issued
            // ahead of this tile's dK/dQ products, so the P^T/dS^T warps find
            // their next scores ready.  With dQ aliasing S^T (d = 128) the next
            // S^T must instead wait for this tile's dQ to be drained.
            if (n_iter > 0) {
                issue_s(0);
                issue_dp(0);
            }
            for (int it = 0; it < n_iter && ok; ++it) {
                const int s = it % QS;
                const uint32_t cur = static_cast<uint32_t>(it) & 1u;
                const uint32_t sQ = sb + L::kQ + s * L::kTile;
                const uint32_t sDO = sb + L::kDO + s * L::kTile;
                // dV += P^T dO
                ok = mbar_wait(bar(L::kPFull), cur, p.status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBlockM / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(sb + L::kPt + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(sDO + kk * 2048, 16384, 1024);
                    mma_bf16_ss(tmem + L::kColDV, a, b, kIdAcc, (it > 0 || kk > 0) ? 1u : 0u);
                }
                if (!L::kDQAliasS && it + 1 < n_iter) issue_s(it + 1);
                if (!ok) break;
                // dK += dS^T Q
                ok = mbar_wait(bar(L::kDSFull), cur, p.status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBlockM / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(sb + L::kDSt + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(sQ + kk * 2048, 16384, 1024);
                    mma_bf16_ss(tmem + L::kColDK, a, b, kIdAcc, (it > 0 || kk > 0) ? 1u : 0u);
                }
                // dQ_t = dS K  (A = dS^T buffer read M-major, B = K read N-major)
                if (!L::kDQAliasS && it >= 1) ok = mbar_wait(bar(L::kDQEmpty), static_cast<uint32_t>(it - 1) & 1u, p.status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(sb + L::kDSt + kk * 2048, 16384, 1024);
                    const uint64_t b = sdesc_sw128(sb + L::kK + kk * 2048, 16384, 1024);
                    mma_bf16_ss(tmem + L::kColDQ, a, b, kIdDQ, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kDQFull));
                mma_commit(bar(L::kQEmpty + s));
                mma_commit(bar(L::kPDSFree));
                if (it + 1 < n_iter) {
                    if (L::kDQAliasS) issue_s(it + 1);
                    issue_dp(it + 1);
                }
            }
            mma_commit(bar(L::kDKVDone));
            mbar_wait(bar(L::kDKVDone), 0, p.status);
        }
    } else {
        // ------------------------- math warpgroups: P^T, dS^T, dQ drain, dK/dV
        const int wg = warp >> 2;             // 0: query columns 0-63, 1: 64-127
        const int wq = warp & 3;              // TMEM lane quarter
        const int kr = threadIdx.x & 127;     // key row within the tile == TMEM lane
        const int c0 = wg * 64;               // first query column of this warpgroup
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
        const uint64_t alx2 = f2_pack(p.scale, p.scale);
        const uint32_t stage = sb + L::kStage + (warp & 7) * 4096;
        bool ok = true;

        // Drain dQ of query tile `jt`: this warp's 32 query rows, this
        // warpgroup's half of the d columns, as 32 x 32 FP32 boxes added into
        // the workspace with TMA reduce-add.
        auto drain_dq = [&](int jt) -> bool {
            bool good = mbar_wait(bar(L::kDQFull), static_cast<uint32_t>(jt) & 1u, p.status);
            if (!__all_sync(0xffffffffu, good)) return false;
            tc_fence_after();
            const int q0 = (qt_begin + jt) * kBlockM;
#pragma unroll
            for (int cb = 0; cb < D / 64; ++cb) {
                const int col = wg * (D / 2) + cb * 32;
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + L::kColDQ + col, r);
                tmem_wait_ld();
                if (cb == D / 64 - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::kDQEmpty));
                }
                if (lane == 0) bulk_wait_read0();  // this warp's previous reduce has read its box
                __syncwarp();
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_shared_v4(stage + sw128_off(lane, ch), r[4 * ch], r[4 * ch + 1], r[4 * ch + 2], r[4 * ch + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_3d(&tm_dqacc, stage, col, q0 + wq * 32, bh);
                    bulk_commit();
                }
            }
            return true;
        };

        for (int it = 0; it < n_iter; ++it) {
            const int s = it % QS;
            const uint32_t u = static_cast<uint32_t>(it / QS);
            const uint32_t cur = static_cast<uint32_t>(it) & 1u;
            const int qt = qt_begin + it;
            if (L::kDQAliasS && it >= 1) {
                // dQ shares the S^T columns: drain it before the next S^T lands
                ok = drain_dq(it - 1);
                if (!ok) break;
            }
            ok = mbar_wait(bar(L::kSFull), cur, p.status) && mbar_wait(bar(L::kQFull + s), u & 1u, p.status);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float4* nl4 = reinterpret_cast<const float4*>(smem + L::kLse + s * 512) + c0 / 4;
            const float4* nd4 = reinterpret_cast<const float4*>(smem + L::kDelta + s * 512) + c0 / 4;
            float pr[64];
            {
                uint32_t r[2][32];
                tmem_ld32(tmem + lane_off + L::kColS + c0, r[0]);
                tmem_ld32(tmem + lane_off + L::kColS + c0 + 32, r[1]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::kSEmpty));
                // P^T[kr][q] = exp2(s * alpha*log2e - LSE_q*log2e)
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    const float4 n = nl4[g];
                    const uint32_t* rr = &r[g >> 3][(g & 7) * 4];
                    float x0, x1, x2, x3;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[0]), __uint_as_float(rr[1])), sl2x2, f2_pack(n.x, n.y)),
                              x0, x1);
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[2]), __uint_as_float(rr[3])), sl2x2, f2_pack(n.z, n.w)),
                              x2, x3);
                    pr[4 * g] = ex2_approx(x0);
                    pr[4 * g + 1] = ex2_approx(x1);
                    pr[4 * g + 2] = ex2_approx(x2);
                    pr[4 * g + 3] = ex2_approx(x3);
                }
            }
            if (CAUSAL && qt == kt) {
                // diagonal tile: query q sees key kr only if q >= kr
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c0 + c < kr) pr[c] = 0.f;
            }
            if (it >= 1) {
                ok = mbar_wait(bar(L::kPDSFree), static_cast<uint32_t>(it - 1) & 1u, p.status);
                if (!ok) break;
            }
            const uint32_t pt_blk = sb + L::kPt + wg * 16384;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const int c = ch * 8;
                st_shared_v4(pt_blk + sw128_off(kr, ch), pack_bf16x2(pr[c], pr[c + 1]), pack_bf16x2(pr[c + 2], pr[c + 3]),
                             pack_bf16x2(pr[c + 4], pr[c + 5]), pack_bf16x2(pr[c + 6], pr[c + 7]));
            }
            fence_async_smem();
            mbar_arrive(bar(L::kPFull));
            if (!L::kDQAliasS && it >= 1) {
                // the previous tile's dQ has been computed meanwhile
                ok = drain_dq(it - 1);
                if (!ok) break;
            }
            // dS^T[kr][q] = P * (alpha * dP + (-alpha * delta_q))
            ok = mbar_wait(bar(L::kDPFull), cur, p.status);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t ds_blk = sb + L::kDSt + wg * 16384;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + L::kColDP + c0 + h * 32, r);
                tmem_wait_ld();
                if (h == 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::kDPEmpty));
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {  // 8 queries per group
                    const int c = h * 32 + g * 8;
                    const float4 na = nd4[c / 4];
                    const float4 nb = nd4[c / 4 + 1];
                    const uint32_t* rr = &r[g * 8];
                    float d[8];
                    f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rr[0]), __uint_as_float(rr[1])), alx2, f2_pack(na.x, na.y)),
                                     f2_pack(pr[c], pr[c + 1])), d[0], d[1]);
                    f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rr[2]), __uint_as_float(rr[3])), alx2, f2_pack(na.z, na.w)),
                                     f2_pack(pr[c + 2], pr[c + 3])), d[2], d[3]);
                    f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rr[4]), __uint_as_float(rr[5])), alx2, f2_pack(nb.x, nb.y)),
                                     f2_pack(pr[c + 4], pr[c + 5])), d[4], d[5]);
                    f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rr[6]), __uint_as_float(rr[7])), alx2, f2_pack(nb.z, nb.w)),
                                     f2_pack(pr[c + 6], pr[c + 7])), d[6], d[7]);
                    st_shared_v4(ds_blk + sw128_off(kr, c >> 3), pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]),
                                 pack_bf16x2(d[4], d[5]), pack_bf16x2(d[6], d[7]));
                }
            }
            fence_async_smem();
            mbar_arrive(bar(L::kDSFull));
        }
        if (ok && n_iter > 0) ok = drain_dq(n_iter - 1);
        if (lane == 0) bulk_wait0();
        // dK, dV epilogue: key rows, this warpgroup's half of the d columns
        if (ok) ok = mbar_wait(bar(L::kDKVDone), 0, p.status);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const int krow = k0 + kr;
            const bool store = krow < p.N;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(which == 0 ? p.dv : p.dk);
                const uint32_t col = (which == 0 ? L::kColDV : L::kColDK) + wg * (D / 2);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_off + col + c * 32, r);
                    tmem_wait_ld();
                    if (!store) continue;
                    uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * p.N + krow) * D + wg * (D / 2) +
                                                          c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]), __uint_as_float(r[8 * e + 1]));
                        w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]), __uint_as_float(r[8 * e + 3]));
                        w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]), __uint_as_float(r[8 * e + 5]));
                        w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]), __uint_as_float(r[8 * e + 7]));
                        dst[e] = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_main(const BwdArgs& a, cudaStream_t stream) {
    using L = BwdLayout<D>;
    auto kern = bwd_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) {
        set_error("bwd_main cudaFuncSetAttribute", e);
        return e;
    }
    BwdParams p;
    p.lse2 = a.lse2;
    p.delta = a.delta;
    p.dk = a.dk;
    p.dv = a.dv;
    p.BH = a.BH;
    p.N = a.N;
    p.Npad = a.Npad;
    p.scale = a.scale;
    p.scale_log2 = a.scale_log2;
    p.status = a.status;
    const int n_kt = (a.N + kBlockN - 1) / kBlockN;
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>(n_kt));
    prof_begin(3, stream);
    kern<<<grid, 320, L::kAlloc, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dqacc, p);
    prof_end(3, stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaFuncAttributes fa_attr{};
        char msg[200];
        if (cudaFuncGetAttributes(&fa_attr, kern) == cudaSuccess)
            snprintf(msg, sizeof msg, "%s (regs %d, max threads %d, local %zu B, dyn smem %d B)",
                     cudaGetErrorString(e), fa_attr.numRegs, fa_attr.maxThreadsPerBlock,
                     fa_attr.localSizeBytes, L::kAlloc);
        else
            snprintf(msg, sizeof msg, "%s", cudaGetErrorString(e));
        set_error_msg("bwd_main launch", msg);
    }
    return e;
}

int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
    const int sms = num_sms();
    prof_begin(2, stream);
    if (a.d == 64)
        bwd_pre_kernel<64><<<sms * 4, 256, 0, stream>>>(a);
    else
        bwd_pre_kernel<128><<<sms * 4, 256, 0, stream>>>(a);
    prof_end(2, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("bwd_pre launch", e);
        return e;
    }
    if (a.d == 64)
        e = a.causal ? launch_main<64, true>(a, stream) : launch_main<64, false>(a, stream);
    else
        e = a.causal ? launch_main<128, true>(a, stream) : launch_main<128, false>(a, stream);
    if (e != cudaSuccess) return e;
    const size_t n8 = static_cast<size_t>(a.BH) * a.N * a.d / 8;
    prof_begin(4, stream);
    dq_convert_kernel<<<sms * 4, 256, 0, stream>>>(a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), n8);
    prof_end(4, stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) set_error("dq_convert launch", e);
    return e;
}

}  // namespace fa
