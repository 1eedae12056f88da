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
// Three kernels, each launched with programmatic dependent launch so that it
// is scheduled while its predecessor finishes (its griddepcontrol.wait still
// waits for the whole predecessor):
//   pre      -LSE*log2(e) and -alpha*delta per row into padded workspaces
//            (delta from the stored O of the mode); on a fresh workspace the
//            same launch clears the FP32 dQ accumulator.
//   main     persistent, one CTA per SM: work items (batch*head, 128-key
//            tile); K and V stay in shared memory while the CTA walks the
//            128-query tiles (causal: only tiles at or below the diagonal).
//            Per query tile, five tcgen05 MMAs:
//              S^T  = K Q^T      (TMEM, FP32)
//              dP^T = V dO^T     (TMEM, FP32)
//              dV  += P^T dO     (TMEM accumulator)
//              dK  += dS^T Q     (TMEM accumulator)
//              dQ_t = dS K       (TMEM), added to the FP32 accumulator with
//                                TMA reduce-add
//            Warp roles: two math warpgroups (warps 0-3: query columns 0-63
//            of the tile, warps 4-7: columns 64-127; thread t of a warpgroup
//            owns key row t) recompute P^T and dS^T; a drain warpgroup (warps
//            8-11, one TMEM lane quarter each) moves each dQ tile from TMEM
//            into the reduce-add and each item's dK and dV from TMEM to HBM
//            (TMA stores), off the math chain; warp 12 issues TMA loads; warp
//            13 issues the MMAs.  The next tile's S^T and dP^T are issued
//            ahead of the current tile's dK/dQ products.
//   convert  the FP32 dQ accumulator to BF16 (and, when asked, zeros written
//            back, leaving the accumulator ready for the next call).
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cstdio>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

struct BwdParams {
    const void* o;        // [BH, N, d] BF16, or FP32 in mode 2
    const float* lse;     // [BH, N]
    const void* dout;     // [BH, N, d] BF16
    float* dq_acc;        // FP32 [BH, N, d] accumulator
    void* dq;             // [BH, N, d] BF16 output
    float* lse2;          // [BH, Npad]: -LSE*log2(e), -inf on padded rows
    float* delta;         // [BH, Npad]: -alpha*rowsum(dO o O), 0 on padded rows
    int delta_given;      // 1: delta already holds -alpha*rowsum(dP o P); pre forms lse2 only
    int zero_acc;         // 1: pre also clears the dQ accumulator
    const float* o32;     // per-head modes: FP32 O of the heads in fp32_mask (o holds the others)
    uint64_t fp32_mask;
    int H;
    RowLayout lay;        // q, k, v, o, dO, dq, dk, dv rows (the tensor maps are 4-D)
    int BH, N, Npad, mode;
    int n_kt;     // key tiles per (batch, head)
    int n_items;  // BH * n_kt
    float scale, scale_log2;
    int* status;
};

constexpr int kBwdThreads = 512;
constexpr int kAuxThreads = 256;   // pre and convert kernels
constexpr int kAuxBlocksPerSM = 8;

// ------------------------------------------------------------------ pre ----
// D/8 threads per row, 8 elements (16 bytes of dO) each; rows padded to Npad.
// Each warp takes kUnroll groups of rows at once, every load of a group (dO,
// O and the LSE) issued before any is used, so that enough loads are in
// flight to keep HBM busy.  O32: O is FP32 (mode 2).  sel < 0: every row;
// sel = 0 / 1: only the rows of heads outside / inside fp32_mask (per-head
// modes), whose O is read from o (BF16) / o32 (FP32).  With zero_acc the
// second half of the blocks clears the dQ accumulator meanwhile.
template <int D, bool O32>
__global__ void __launch_bounds__(kAuxThreads) bwd_pre_kernel(const BwdParams p, int sel) {
    constexpr int TPR = D / 8;       // threads per row
    constexpr int RPW = 32 / TPR;    // rows per warp and group
    constexpr int kUnroll = O32 ? 3 : 4;
    // the next kernel may be scheduled now; it waits for this one to finish
    griddep_launch_dependents();
    const int row_blocks = p.zero_acc ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
    if (static_cast<int>(blockIdx.x) >= row_blocks) {
        // the previous user of this workspace's memory must be done
        griddep_wait();
        const size_t n4 = static_cast<size_t>(p.BH) * p.N * D / 4;
        float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
        const size_t nthr = static_cast<size_t>(gridDim.x - row_blocks) * blockDim.x;
        const size_t tid = static_cast<size_t>(blockIdx.x - row_blocks) * blockDim.x + threadIdx.x;
        for (size_t e = tid; e < n4; e += 4 * nthr) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (e + u * nthr < n4) acc4[e + u * nthr] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const void* obase = (sel == 1) ? static_cast<const void*>(p.o32) : p.o;
    const int lane = threadIdx.x & 31;
    const int sub = lane % TPR;
    // rows < 2^31 (BH * Npad * d is checked against it), so 32-bit index math
    const int rows = p.BH * p.Npad;
    const int nwarps = row_blocks * (blockDim.x >> 5);
    const int gw = static_cast<int>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const float log2e = 1.4426950408889634f;
    bool waited = false;
    for (int r0 = gw * RPW * kUnroll; r0 < rows; r0 += nwarps * RPW * kUnroll) {
        uint4 g[kUnroll], o[kUnroll], o2[kUnroll];
        float lse[kUnroll];
        bool valid[kUnroll], chosen[kUnroll];
        size_t rowi[kUnroll], base[kUnroll];
        // dO is an input of the call, not an output of the previous kernel:
        // its loads are issued before the wait for that kernel
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int r = r0 + u * RPW + lane / TPR;
            const int bh = r / p.Npad;
            const int i = r - bh * p.Npad;
            chosen[u] = r < rows && (sel < 0 || static_cast<int>((p.fp32_mask >> (bh % p.H)) & 1ull) == sel);
            valid[u] = chosen[u] && i < p.N;
            g[u] = o[u] = o2[u] = make_uint4(0u, 0u, 0u, 0u);
            lse[u] = 0.f;
            rowi[u] = static_cast<size_t>(bh) * p.N + i;
            base[u] = (p.lay.head_inner ? p.lay.row(bh, i) : rowi[u] * D) + sub * 8;
            if (valid[u] && !p.delta_given)
                g[u] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + base[u]);
        }
        // O and the LSE come from the previous kernel (the forward); this
        // launch's writes below must also follow it
        if (!waited) {
            griddep_wait();
            waited = true;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (valid[u]) {
                if (sub == 0) lse[u] = p.lse[rowi[u]];
                if (!p.delta_given) {
                    if (O32) {
                        o[u] = *reinterpret_cast<const uint4*>(static_cast<const float*>(obase) + base[u]);
                        o2[u] = *reinterpret_cast<const uint4*>(static_cast<const float*>(obase) + base[u] + 4);
                    } else {
                        o[u] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(obase) + base[u]);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t gw4[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
            float acc = 0.f;
            if (O32) {
                const uint32_t of[8] = {o[u].x, o[u].y, o[u].z, o[u].w, o2[u].x, o2[u].y, o2[u].z, o2[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(__uint_as_float(gw4[e] << 16), __uint_as_float(of[2 * e]), acc);
                    acc = fmaf(__uint_as_float(gw4[e] & 0xFFFF0000u), __uint_as_float(of[2 * e + 1]), acc);
                }
            } else {
                const uint32_t ow4[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(__uint_as_float(gw4[e] << 16), __uint_as_float(ow4[e] << 16), acc);
                    acc = fmaf(__uint_as_float(gw4[e] & 0xFFFF0000u), __uint_as_float(ow4[e] & 0xFFFF0000u), acc);
                }
            }
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const int r = r0 + u * RPW + lane / TPR;
            if (sub == 0 && chosen[u]) {
                // stored pre-negated / pre-scaled for the main kernel's FMAs:
                //   P  = exp2(s * alpha*log2e + lse2),  lse2 = -LSE*log2e
                //   dS = P * (alpha * dP + delta),      delta = -alpha * rowsum(dO o O)
                if (!p.delta_given) p.delta[r] = valid[u] ? -p.scale * acc : 0.f;
                // padded rows: P = exp2(s - inf) = 0
                p.lse2[r] = valid[u] ? -lse[u] * log2e : -INFINITY;
            }
        }
    }
}

// -------------------------------------------------------------- convert ----
// dQ accumulator (FP32) -> BF16 in the caller's layout, eight elements per
// thread and step, four steps' loads in flight.
template <int D>
__global__ void __launch_bounds__(kAuxThreads) dq_convert_kernel(const BwdParams p) {
    constexpr int kChunks = D / 8;  // eight-element chunks per row
    griddep_launch_dependents();
    griddep_wait();  // every reduce-add of the main kernel has landed
    const float4* acc = reinterpret_cast<const float4*>(p.dq_acc);
    uint4* dq = reinterpret_cast<uint4*>(p.dq);
    // BH * Npad * d < 2^31 (checked on the host): 32-bit chunk indices
    const int n8 = p.BH * p.N * kChunks;
    const int nthr = static_cast<int>(gridDim.x * blockDim.x);
    const int tid = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    for (int e0 = tid; e0 < n8; e0 += 4 * nthr) {
        float4 x[4], y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * nthr;
            if (e < n8) {
                x[u] = acc[2 * static_cast<size_t>(e)];
                y[u] = acc[2 * static_cast<size_t>(e) + 1];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * nthr;
            if (e < n8) {
                uint4 w;
                w.x = pack_bf16x2(x[u].x, x[u].y);
                w.y = pack_bf16x2(x[u].z, x[u].w);
                w.z = pack_bf16x2(y[u].x, y[u].y);
                w.w = pack_bf16x2(y[u].z, y[u].w);
                // chunk e of the [BH, N, d] accumulator -> dq in the caller's layout
                size_t dst = static_cast<size_t>(e);
                if (p.lay.head_inner) {
                    const int row = e / kChunks;
                    const int bh = row / p.N;
                    dst = (p.lay.row(bh, row - bh * p.N) >> 3) + static_cast<size_t>(e - row * kChunks);
                }
                dq[dst] = w;
            }
        }
    }
}

// ---------------------------------------------------------------- main ----

template <int D>
struct BwdLayout {
    static constexpr int kTile = kBlockM * D * 2;      // 128 rows x D BF16
    // d = 64: three Q/dO stages, so the next query tile's S^T can be issued
    // while the current one is still being worked on
    static constexpr int kQStages = (D == 64) ? 3 : 1;
    // d = 64: P^T goes to TMEM as the A operand of dV (as Pbar does in the
    // forward), which frees the shared memory for a second K/V buffer: the
    // next work item's K and V load while the current one finishes.
    static constexpr bool kPtInTmem = (D == 64);
    static constexpr int kKVBufs = (D == 64) ? 2 : 1;
    static constexpr int kK = 0;                                  // [kKVBufs]
    static constexpr int kV = kK + kKVBufs * kTile;               // [kKVBufs]
    static constexpr int kQ = kV + kKVBufs * kTile;               // [kQStages]
    static constexpr int kDO = kQ + kQStages * kTile;             // [kQStages]
    static constexpr int kPt = kDO + kQStages * kTile;            // d = 128: 128 keys x 128 queries BF16
    static constexpr int kDSt = kPt + (kPtInTmem ? 0 : kBlockM * kBlockN * 2);
    static constexpr int kStage = kDSt + kBlockM * kBlockN * 2;   // 4 drain warps x (32 x 32 FP32), swizzled
    static constexpr int kLse = kStage + 4 * 4096;                // [kQStages][128] FP32 (-LSE*log2e)
    static constexpr int kDelta = kLse + kQStages * 512;          // [kQStages][128] FP32 (-alpha*delta)
    static constexpr int kBar = kDelta + kQStages * 512;
    // barriers
    static constexpr int kKVFull = 0;                         // [kKVBufs]
    static constexpr int kKVEmpty = kKVFull + kKVBufs;        // [kKVBufs]
    static constexpr int kQFull = kKVEmpty + kKVBufs;         // [kQStages]
    static constexpr int kQEmpty = kQFull + kQStages;         // [kQStages]
    static constexpr int kSFull = kQEmpty + kQStages;
    static constexpr int kSEmpty = kSFull + 1;
    static constexpr int kDPFull = kSEmpty + 1;
    static constexpr int kDPEmpty = kDPFull + 1;
    static constexpr int kPFull = kDPEmpty + 1;
    static constexpr int kDSFull = kPFull + 1;
    static constexpr int kPDSFree = kDSFull + 1;     // the tile's dK and dQ products have read dS^T
    static constexpr int kPtFree = kPDSFree + 1;     // the tile's dV product has read P^T
    static constexpr int kDQFull = kPtFree + 1;
    static constexpr int kDQEmpty = kDQFull + 1;
    static constexpr int kAccDone = kDQEmpty + 1;    // dK, dV of the item complete
    static constexpr int kAccFree = kAccDone + 1;    // dK, dV read out of TMEM
    static constexpr int kDrain = kAccFree + 1;
    static constexpr int kNumBars = kDrain + 1;
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
    static constexpr uint32_t kColPt = 256 + 3 * D;  // d = 64: P^T as BF16 pairs, 64 columns
    static_assert(!kPtInTmem || kColPt + 64 <= 512, "TMEM budget");
    static constexpr uint32_t kMathThreads = 256;  // two warpgroups
    static constexpr uint32_t kDrainThreads = 128; // one warpgroup
    static constexpr int kDrainWarp0 = 8;
    static constexpr int kProducerWarp = 12;
    static constexpr int kMmaWarp = 13;            // warps 14, 15 idle (whole warpgroups for setmaxnreg)
    static constexpr int kThreads = kBwdThreads;
    // registers: 2 x 128 x 168 (math) + 2 x 128 x 88 (drain, producer, MMA) = 512 x 128
    static constexpr uint32_t kRegsMath = 168;
    static constexpr uint32_t kRegsOther = 88;
    static_assert(256 * kRegsMath + 256 * kRegsOther == kThreads * 128, "register split");
};

// Work items are (key tile, batch-head) pairs numbered longest first (causal:
// key tile 0 sees every query tile).  The host assigns them to the CTAs by
// longest-processing-time-first list scheduling: each item in turn, longest
// first, goes to the CTA with the fewest query tiles so far.  For 96 causal
// heads of 8 key tiles on 152 SMs the busiest SM then gets 23 query tiles; a
// snake order over rounds of the grid gives it 24.  items[start[c] ..
// start[c + 1]) are CTA c's items in the order it runs them.  n = 0 (more
// items or CTAs than the table holds): snake order.
constexpr int kSchedMaxCta = 160;
constexpr int kSchedMaxItems = 4096;
struct BwdSched {
    int n;
    uint16_t start[kSchedMaxCta + 1];
    uint16_t items[kSchedMaxItems];
};

// The item CTA blockIdx.x runs in its round r, or INT_MAX past its last.
__device__ __forceinline__ int bwd_item(const BwdSched& sc, int r) {
    const int c = static_cast<int>(blockIdx.x);
    if (sc.n > 0) {
        const int b = sc.start[c], e = sc.start[c + 1];
        return r < e - b ? static_cast<int>(sc.items[b + r]) : INT_MAX;
    }
    const int G = static_cast<int>(gridDim.x);
    return r * G + ((r & 1) ? G - 1 - c : c);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdLayout<D>::kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqacc, const __grid_constant__ CUtensorMap tm_dk,
               const __grid_constant__ CUtensorMap tm_dv, const BwdParams p,
               const __grid_constant__ BwdSched sched) {
    using L = BwdLayout<D>;
    constexpr int QS = L::kQStages;
    constexpr int KVB = L::kKVBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + L::kBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_qt_all = (p.N + kBlockM - 1) / kBlockM;
    auto item_bh = [&](int it) { return it % p.BH; };
    auto item_kt = [&](int it) { return it / p.BH; };
    auto item_qt0 = [&](int kt) { return CAUSAL ? kt : 0; };          // first query tile
    auto item_iters = [&](int kt) { return n_qt_all - item_qt0(kt); };  // query tiles visited

    if (threadIdx.x == 0) {
        for (int b = 0; b < KVB; ++b) {
            mbar_init(bar(L::kKVFull + b), 1);
            mbar_init(bar(L::kKVEmpty + b), 1);
        }
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
        mbar_init(bar(L::kPtFree), 1);
        mbar_init(bar(L::kDQFull), 1);
        mbar_init(bar(L::kDQEmpty), L::kDrainThreads);
        mbar_init(bar(L::kAccDone), 1);
        mbar_init(bar(L::kAccFree), L::kDrainThreads);
        mbar_init(bar(L::kDrain), 1);
        fence_mbar_init();
    }
    if (warp == L::kMmaWarp) {
        tmem_alloc(sb + L::kTmemSlot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

    // Nothing above reads or writes global memory, so under programmatic
    // dependent launch all of it overlaps the previous kernel (pre); the
    // next one (convert) may be scheduled as this grid's CTAs leave.  Every
    // thread but the producer waits for pre here; the producer first issues
    // its first tiles of K, V, Q and dO (inputs of the call, which pre does
    // not write) and waits before the per-row terms that pre writes.
    if (warp != L::kProducerWarp) griddep_wait();
    griddep_launch_dependents();

    if (warp >= L::kDrainWarp0) {
    regs_dec<L::kRegsOther>();
    if (warp == L::kProducerWarp) {
        // -------------------------------------------------------- producer
        // Per item: K and V (into the item's K/V buffer), then Q, dO and the
        // per-row LSE/delta of each query tile through the Q ring, running
        // ahead into the next item as far as the buffers allow.
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            bool ok = true;
            bool waited = false;  // griddepcontrol.wait done (before the first per-row load)
            int g = 0;  // query tiles loaded so far (all items)
            int n = 0;  // items started
            for (int r = 0; ok; ++r, ++n) {
                const int itm = bwd_item(sched, r);
                if (itm >= p.n_items) break;
                const int bh = item_bh(itm), kt = item_kt(itm);
                const int hh = bh % p.H, bb = bh / p.H;  // head and batch of the tile coordinates
                const int kb = n % KVB;
                if (n >= KVB) ok = mbar_wait(bar(L::kKVEmpty + kb), static_cast<uint32_t>(n / KVB - 1) & 1u, p.status);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(L::kKVFull + kb), 2 * L::kTile);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_rows(sb + L::kK + kb * L::kTile + b * 16384, &tm_k, bar(L::kKVFull + kb), b * 64,
                                kt * kBlockN, hh, bb, p.lay.head_inner);
                    tma_load_rows(sb + L::kV + kb * L::kTile + b * 16384, &tm_v, bar(L::kKVFull + kb), b * 64,
                                kt * kBlockN, hh, bb, p.lay.head_inner);
                }
                const int n_iter = item_iters(kt);
                for (int it = 0; it < n_iter; ++it, ++g) {
                    const int s = g % QS;
                    const uint32_t u = static_cast<uint32_t>(g / QS);
                    if (g >= QS && !(ok = mbar_wait(bar(L::kQEmpty + s), (u - 1) & 1u, p.status))) break;
                    const int q0 = (item_qt0(kt) + it) * kBlockM;
                    mbar_arrive_expect_tx(bar(L::kQFull + s), 2 * L::kTile + 1024);
                    for (int b = 0; b < D / 64; ++b) {
                        tma_load_rows(sb + L::kQ + s * L::kTile + b * 16384, &tm_q, bar(L::kQFull + s), b * 64, q0,
                                      hh, bb, p.lay.head_inner);
                        tma_load_rows(sb + L::kDO + s * L::kTile + b * 16384, &tm_do, bar(L::kQFull + s), b * 64, q0,
                                      hh, bb, p.lay.head_inner);
                    }
                    const size_t roff = static_cast<size_t>(bh) * p.Npad + q0;
                    if (!waited) {
                        griddep_wait();
                        waited = true;
                    }
                    bulk_load(sb + L::kLse + s * 512, p.lse2 + roff, 512, bar(L::kQFull + s));
                    bulk_load(sb + L::kDelta + s * 512, p.delta + roff, 512, bar(L::kQFull + s));
                }
            }
            // Every copy this thread issued must have landed before the CTA
            // may exit (normally long since true).
            for (int m = n - KVB > 0 ? n - KVB : 0; m < n; ++m)
                mbar_wait(bar(L::kKVFull + m % KVB), static_cast<uint32_t>(m / KVB) & 1u, p.status);
            for (int h = g - QS > 0 ? g - QS : 0; h < g; ++h)
                mbar_wait(bar(L::kQFull + h % QS), static_cast<uint32_t>(h / QS) & 1u, p.status);
        }
    } else if (warp == L::kMmaWarp) {
        // ------------------------------------------------------ MMA issuer
        // The whole warp runs the loop and waits; one elected lane issues each
        // group of MMAs together with the commits that track them.
        constexpr uint32_t kIdSS = idesc_bf16(kBlockM, kBlockN, false, false);  // S^T, dP^T
        constexpr uint32_t kIdAcc = idesc_bf16(kBlockM, D, false, true);         // dV, dK
        constexpr uint32_t kIdDQ = idesc_bf16(kBlockM, D, true, true);           // dQ
        auto wait_all = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, p.status));
        };
        bool ok = true;
        bool issued = false;
        // S^T(gi) = K Q^T with the K tile at sK
        auto issue_s = [&](int gi, uint32_t sK) {
            const int s = gi % QS;
            ok = ok && wait_all(bar(L::kQFull + s), static_cast<uint32_t>(gi / QS) & 1u);
            if (ok && gi >= 1) ok = wait_all(bar(L::kSEmpty), static_cast<uint32_t>(gi - 1) & 1u);
            if (ok && gi >= 1 && L::kDQAliasS) ok = wait_all(bar(L::kDQEmpty), static_cast<uint32_t>(gi - 1) & 1u);
            if (!ok) return;
            tc_fence_after();
            const uint32_t sQ = sb + L::kQ + s * L::kTile;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16_ss(tmem + L::kColS, sdesc_sw128(sK + ko, 16, 1024), sdesc_sw128(sQ + ko, 16, 1024),
                                kIdSS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kSFull));
            }
            __syncwarp();
            issued = true;
        };
        // dP^T(gi) = V dO^T with the V tile at sV (Q/dO stage gi is already known to be loaded)
        auto issue_dp = [&](int gi, uint32_t sV) {
            const int s = gi % QS;
            if (ok && gi >= 1) ok = wait_all(bar(L::kDPEmpty), static_cast<uint32_t>(gi - 1) & 1u);
            if (!ok) return;
            tc_fence_after();
            const uint32_t sDO = sb + L::kDO + s * L::kTile;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16_ss(tmem + L::kColDP, sdesc_sw128(sV + ko, 16, 1024), sdesc_sw128(sDO + ko, 16, 1024),
                                kIdSS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kDPFull));
            }
            __syncwarp();
        };
        // Software pipeline: the next tile's S^T is issued as soon as the math
        // warps have read this tile's S^T, and the next dP^T as soon as they
        // have read this dP^T, so both are ready before the math warps ask.
        // The next tile may belong to the next item (its K/V sit in the other
        // buffer), so items follow one another without a bubble.  With dQ
        // aliasing S^T (d = 128, one K/V buffer) the next S^T must instead wait
        // for this tile's dQ to be drained, after the dQ product, and a new
        // item starts only after the previous one's products.
        int g = 0;  // query tiles processed so far (all items)
        int itm = bwd_item(sched, 0);
        bool head_issued = false;  // this item's first S^T/dP^T already issued
        for (int r = 0, n = 0; ok && itm < p.n_items; ++r, ++n) {
            const int kt = item_kt(itm);
            const int n_iter = item_iters(kt);
            const int kb = n % KVB;
            const uint32_t sK = sb + L::kK + kb * L::kTile;
            const uint32_t sV = sb + L::kV + kb * L::kTile;
            const int itm_next = bwd_item(sched, r + 1);
            const bool has_next = itm_next < p.n_items;
            const uint32_t sK_next = sb + L::kK + ((n + 1) % KVB) * L::kTile;
            const uint32_t sV_next = sb + L::kV + ((n + 1) % KVB) * L::kTile;
            if (!head_issued) {
                ok = wait_all(bar(L::kKVFull + kb), static_cast<uint32_t>(n / KVB) & 1u);
                if (!ok) break;
                issue_s(g, sK);
                issue_dp(g, sV);
            }
            head_issued = false;
            for (int it = 0; it < n_iter && ok; ++it, ++g) {
                const int s = g % QS;
                const uint32_t cur = static_cast<uint32_t>(g) & 1u;
                const uint32_t sQ = sb + L::kQ + s * L::kTile;
                const uint32_t sDO = sb + L::kDO + s * L::kTile;
                const bool last = (it + 1 == n_iter);
                // the next tile (of this item, or the next item's first)
                const bool ahead = !L::kDQAliasS && (!last || has_next);
                if (ahead) {
                    if (last) ok = wait_all(bar(L::kKVFull + (n + 1) % KVB), static_cast<uint32_t>((n + 1) / KVB) & 1u);
                    issue_s(g + 1, last ? sK_next : sK);
                }
                // dV += P^T dO; the item's first product overwrites dV, which
                // the previous item's epilogue must have read out
                ok = ok && wait_all(bar(L::kPFull), cur);
                if (ok && it == 0 && n >= 1) ok = wait_all(bar(L::kAccFree), static_cast<uint32_t>(n - 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBlockM / 16; ++kk) {
                        const uint64_t b = sdesc_sw128(sDO + kk * 2048, 16384, 1024);
                        if (L::kPtInTmem) {
                            mma_bf16_ts(tmem + L::kColDV, tmem + L::kColPt + kk * 8, b, kIdAcc, (it > 0 || kk > 0) ? 1u : 0u);
                        } else {
                            const uint64_t a = sdesc_sw128(sb + L::kPt + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                            mma_bf16_ss(tmem + L::kColDV, a, b, kIdAcc, (it > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    // P^T may be overwritten once dV has read it, well
                    // before this tile's dK and dQ are done with dS^T
                    mma_commit(bar(L::kPtFree));
                }
                __syncwarp();
                if (ahead) {
                    issue_dp(g + 1, last ? sV_next : sV);
                    if (last) head_issued = true;
                }
                if (!ok) break;
                // dK += dS^T Q
                ok = wait_all(bar(L::kDSFull), cur);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBlockM / 16; ++kk) {
                        const uint64_t a = sdesc_sw128(sb + L::kDSt + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(sQ + kk * 2048, 16384, 1024);
                        mma_bf16_ss(tmem + L::kColDK, a, b, kIdAcc, (it > 0 || kk > 0) ? 1u : 0u);
                    }
                    // d = 128 (a single Q/dO stage, so the next tile's load
                    // waits for this release): the stage's last readers (S^T,
                    // dP^T, dV, dK) are issued, so release it before the dQ
                    // product, which reads only dS^T and K
                    if (L::kQStages == 1) mma_commit(bar(L::kQEmpty + s));
                }
                __syncwarp();
                // dQ_t = dS K  (A = dS^T buffer read M-major, B = K read N-major)
                if (!L::kDQAliasS && g >= 1) ok = wait_all(bar(L::kDQEmpty), static_cast<uint32_t>(g - 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk) {
                        const uint64_t a = sdesc_sw128(sb + L::kDSt + kk * 2048, 16384, 1024);
                        const uint64_t b = sdesc_sw128(sK + kk * 2048, 16384, 1024);
                        mma_bf16_ss(tmem + L::kColDQ, a, b, kIdDQ, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(L::kDQFull));
                    if (L::kQStages > 1) mma_commit(bar(L::kQEmpty + s));
                    mma_commit(bar(L::kPDSFree));
                    if (last) {
                        mma_commit(bar(L::kKVEmpty + kb));  // last read of this item's K and V
                        mma_commit(bar(L::kAccDone));
                    }
                }
                __syncwarp();
                if (L::kDQAliasS && !last) {
                    issue_s(g + 1, sK);
                    issue_dp(g + 1, sV);
                }
            }
            itm = itm_next;
        }
        // Drain: every MMA this warp issued has completed before TMEM is freed.
        if (issued) {
            if (elect_one()) mma_commit(bar(L::kDrain));
            __syncwarp();
            mbar_wait(bar(L::kDrain), 0, p.status);
        }
    } else if (warp < L::kDrainWarp0 + 4) {
        // ------------------------------------------------- dQ drain warpgroup
        // Per query tile: this warp's 32 query rows (its TMEM lane quarter) of
        // dQ, read out of TMEM 64 columns at a time, staged as 32 x 32 FP32
        // boxes (one buffer per warp) and added into the workspace with TMA
        // reduce-add.  The tile's TMEM columns are released as soon as the last
        // columns are in registers.
        const int wq = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t stg = sb + L::kStage + wq * 4096;
        auto wait_w = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, p.status));
        };
        bool ok = true;
        int g = 0;  // query tiles so far (all items)
        for (int r = 0, n = 0; ok; ++r, ++n) {
            const int itm = bwd_item(sched, r);
            if (itm >= p.n_items) break;
            const int bh = item_bh(itm), kt = item_kt(itm);
            const int hh = bh % p.H, bb = bh / p.H;  // head and batch of the tile coordinates
            const int n_iter = item_iters(kt);
            for (int it = 0; it < n_iter; ++it, ++g) {
                ok = wait_w(bar(L::kDQFull), static_cast<uint32_t>(g) & 1u);
                if (!ok) break;
                tc_fence_after();
                const int q0 = (item_qt0(kt) + it) * kBlockM;
#pragma unroll
                for (int pr2 = 0; pr2 < D / 64; ++pr2) {
                    uint32_t rv[2][32];
                    tmem_ld32(tmem + lane_off + L::kColDQ + pr2 * 64, rv[0]);
                    tmem_ld32(tmem + lane_off + L::kColDQ + pr2 * 64 + 32, rv[1]);
                    tmem_wait_ld();
                    if (pr2 == D / 64 - 1) {
                        tc_fence_before();
                        mbar_arrive(bar(L::kDQEmpty));
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (lane == 0) bulk_wait_read0();  // the previous reduce has read the buffer
                        __syncwarp();
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            st_shared_v4(stg + sw128_off(lane, ch), rv[h][4 * ch], rv[h][4 * ch + 1], rv[h][4 * ch + 2],
                                         rv[h][4 * ch + 3]);
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_3d(&tm_dqacc, stg, pr2 * 64 + h * 32, q0 + wq * 32, bh);
                            bulk_commit();
                        }
                    }
                }
            }
            if (!ok) break;
            // -------------------------------------------- dK/dV epilogue
            // This warp's 32 key rows of dV and dK: read out of TMEM (which
            // frees the accumulators for the next item's first products),
            // staged as BF16 in the 128-byte-swizzled box layout (64 columns x
            // 32 rows, 4 KB) and written by TMA; rows past N are clipped.
            ok = wait_w(bar(L::kAccDone), static_cast<uint32_t>(n) & 1u);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
#pragma unroll
                for (int b64 = 0; b64 < D / 64; ++b64) {
                    uint32_t av[2][32];
                    const uint32_t col = (which == 0 ? L::kColDV : L::kColDK) + b64 * 64;
                    tmem_ld32(tmem + lane_off + col, av[0]);
                    tmem_ld32(tmem + lane_off + col + 32, av[1]);
                    tmem_wait_ld();
                    if (which == 1 && b64 == D / 64 - 1) {
                        tc_fence_before();
                        mbar_arrive(bar(L::kAccFree));
                    }
                    if (lane == 0) bulk_wait_read0();  // the previous store or reduce has read the buffer
                    __syncwarp();
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(stg + sw128_off(lane, ch),
                                     pack_bf16x2(__uint_as_float(av[ch >> 2][(ch & 3) * 8 + 0]), __uint_as_float(av[ch >> 2][(ch & 3) * 8 + 1])),
                                     pack_bf16x2(__uint_as_float(av[ch >> 2][(ch & 3) * 8 + 2]), __uint_as_float(av[ch >> 2][(ch & 3) * 8 + 3])),
                                     pack_bf16x2(__uint_as_float(av[ch >> 2][(ch & 3) * 8 + 4]), __uint_as_float(av[ch >> 2][(ch & 3) * 8 + 5])),
                                     pack_bf16x2(__uint_as_float(av[ch >> 2][(ch & 3) * 8 + 6]), __uint_as_float(av[ch >> 2][(ch & 3) * 8 + 7])));
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_rows(which == 0 ? &tm_dv : &tm_dk, stg, b64 * 64, kt * kBlockN + wq * 32, hh, bb, p.lay.head_inner);
                        bulk_commit();
                    }
                }
            }
        }
        // every reduce-add and store has landed (not only read its staging
        // buffer) before the CTA exits
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }
    } else {
    regs_inc<L::kRegsMath>();
    {
        // ------------------------- math warpgroups: P^T, dS^T, dK/dV
        const int wg = warp >> 2;             // 0: query columns 0-63, 1: 64-127
        const int wq = warp & 3;              // TMEM lane quarter
        const int kr = threadIdx.x & 127;     // key row within the tile == TMEM lane
        const int c0 = wg * 64;               // first query column of this warpgroup
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
        const uint64_t alx2 = f2_pack(p.scale, p.scale);
        auto wait_w = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, p.status));
        };
        bool ok = true;
        int g = 0;  // query tiles processed so far (all items)

        for (int r = 0; ok; ++r) {
            const int itm = bwd_item(sched, r);
            if (itm >= p.n_items) break;
            const int kt = item_kt(itm);
            const int qt_begin = item_qt0(kt);
            const int n_iter = item_iters(kt);
            for (int it = 0; it < n_iter; ++it, ++g) {
                const int s = g % QS;
                const uint32_t u = static_cast<uint32_t>(g / QS);
                const uint32_t cur = static_cast<uint32_t>(g) & 1u;
                const int qt = qt_begin + it;
                ok = wait_w(bar(L::kSFull), cur) && wait_w(bar(L::kQFull + s), u & 1u);
                if (!ok) break;
                tc_fence_after();
                const float4* nl4 = reinterpret_cast<const float4*>(smem + L::kLse + s * 512) + c0 / 4;
                const float4* nd4 = reinterpret_cast<const float4*>(smem + L::kDelta + s * 512) + c0 / 4;
                float pr[64];
                {
                    uint32_t rr2[2][32];
                    tmem_ld32(tmem + lane_off + L::kColS + c0, rr2[0]);
                    tmem_ld32(tmem + lane_off + L::kColS + c0 + 32, rr2[1]);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(L::kSEmpty));
                    // P^T[kr][q] = exp2(s * alpha*log2e - LSE_q*log2e)
#pragma unroll
                    for (int gg = 0; gg < 16; ++gg) {
                        const float4 nv = nl4[gg];
                        const uint32_t* rr = &rr2[gg >> 3][(gg & 7) * 4];
                        float x0, x1, x2, x3;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[0]), __uint_as_float(rr[1])), sl2x2,
                                         f2_pack(nv.x, nv.y)),
                                  x0, x1);
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[2]), __uint_as_float(rr[3])), sl2x2,
                                         f2_pack(nv.z, nv.w)),
                                  x2, x3);
                        pr[4 * gg] = ex2_approx(x0);
                        pr[4 * gg + 1] = ex2_approx(x1);
                        pr[4 * gg + 2] = ex2_approx(x2);
                        pr[4 * gg + 3] = ex2_approx(x3);
                    }
                }
                if (CAUSAL && qt == kt) {
                    // diagonal tile: query q sees key kr only if q >= kr
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c0 + c < kr) pr[c] = 0.f;
                }
                // P^T overwrites the previous tile's, which its dV product reads
                if (g >= 1) {
                    ok = wait_w(bar(L::kPtFree), static_cast<uint32_t>(g - 1) & 1u);
                    if (!ok) break;
                }
                if (L::kPtInTmem) {
                    uint32_t w[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) w[e] = pack_bf16x2(pr[2 * e], pr[2 * e + 1]);
                    tmem_st32(tmem + lane_off + L::kColPt + wg * 32, w);
                    tmem_wait_st();
                    tc_fence_before();
                } else {
                    const uint32_t pt_blk = sb + L::kPt + wg * 16384;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const int c = ch * 8;
                        st_shared_v4(pt_blk + sw128_off(kr, ch), pack_bf16x2(pr[c], pr[c + 1]),
                                     pack_bf16x2(pr[c + 2], pr[c + 3]), pack_bf16x2(pr[c + 4], pr[c + 5]),
                                     pack_bf16x2(pr[c + 6], pr[c + 7]));
                    }
                    fence_async_smem();
                }
                mbar_arrive(bar(L::kPFull));
                // dS^T[kr][q] = P * (alpha * dP + (-alpha * delta_q))
                ok = wait_w(bar(L::kDPFull), cur);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ds_blk = sb + L::kDSt + wg * 16384;
                uint32_t dpr[2][32];
                tmem_ld32(tmem + lane_off + L::kColDP + c0, dpr[0]);
                tmem_ld32(tmem + lane_off + L::kColDP + c0 + 32, dpr[1]);
                tmem_wait_ld();  // one wait for both loads
                tc_fence_before();
                mbar_arrive(bar(L::kDPEmpty));
                // dS^T into the registers that held P^T, then stored once the
                // previous tile's dK and dQ products have read dS^T
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq) {  // 8 queries per group
                        const int c = h * 32 + gq * 8;
                        const float4 na = nd4[c / 4];
                        const float4 nb = nd4[c / 4 + 1];
                        const uint32_t* rv = &dpr[h][gq * 8];
                        f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rv[0]), __uint_as_float(rv[1])), alx2,
                                                f2_pack(na.x, na.y)),
                                         f2_pack(pr[c], pr[c + 1])),
                                  pr[c], pr[c + 1]);
                        f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rv[2]), __uint_as_float(rv[3])), alx2,
                                                f2_pack(na.z, na.w)),
                                         f2_pack(pr[c + 2], pr[c + 3])),
                                  pr[c + 2], pr[c + 3]);
                        f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rv[4]), __uint_as_float(rv[5])), alx2,
                                                f2_pack(nb.x, nb.y)),
                                         f2_pack(pr[c + 4], pr[c + 5])),
                                  pr[c + 4], pr[c + 5]);
                        f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(rv[6]), __uint_as_float(rv[7])), alx2,
                                                f2_pack(nb.z, nb.w)),
                                         f2_pack(pr[c + 6], pr[c + 7])),
                                  pr[c + 6], pr[c + 7]);
                    }
                }
                if (g >= 1) {
                    ok = wait_w(bar(L::kPDSFree), static_cast<uint32_t>(g - 1) & 1u);
                    if (!ok) break;
                }
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const int c = ch * 8;
                    st_shared_v4(ds_blk + sw128_off(kr, ch), pack_bf16x2(pr[c], pr[c + 1]), pack_bf16x2(pr[c + 2], pr[c + 3]),
                                 pack_bf16x2(pr[c + 4], pr[c + 5]), pack_bf16x2(pr[c + 6], pr[c + 7]));
                }
                fence_async_smem();
                mbar_arrive(bar(L::kDSFull));
            }
        }
    }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == L::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

BwdParams make_params(const BwdArgs& a) {
    BwdParams p;
    p.o = a.o;
    p.lse = a.lse;
    p.dout = a.dout;
    p.dq_acc = a.dq_acc;
    p.dq = a.dq;
    p.lse2 = a.lse2;
    p.delta = a.delta;
    p.delta_given = a.delta_given;
    p.zero_acc = a.zero_acc;
    p.o32 = a.o32;
    p.fp32_mask = a.fp32_mask;
    p.H = a.lay.H;
    p.lay = a.lay;
    p.mode = a.mode;
    p.BH = a.BH;
    p.N = a.N;
    p.Npad = a.Npad;
    p.n_kt = (a.N + kBlockN - 1) / kBlockN;
    p.n_items = a.BH * p.n_kt;
    p.scale = a.scale;
    p.scale_log2 = a.scale_log2;
    p.status = a.status;
    return p;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream finishes; its griddepcontrol.wait
// holds it until that kernel is complete.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, int threads, int smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

template <int D>
cudaError_t launch_pre(const BwdParams& p, int num_sms, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(num_sms * kAuxBlocksPerSM));
    cudaError_t e = cudaSuccess;
    prof_begin(2, stream);
    if (p.fp32_mask != 0) {  // per-head modes: each head's delta from its own stored O
        BwdParams p1 = p;
        p1.zero_acc = 0;     // the first launch clears the accumulator
        e = launch_pdl(bwd_pre_kernel<D, false>, grid, kAuxThreads, 0, stream, p, 0);
        if (e == cudaSuccess) e = launch_pdl(bwd_pre_kernel<D, true>, grid, kAuxThreads, 0, stream, p1, 1);
    } else if (p.mode == 2) {
        e = launch_pdl(bwd_pre_kernel<D, true>, grid, kAuxThreads, 0, stream, p, -1);
    } else {
        e = launch_pdl(bwd_pre_kernel<D, false>, grid, kAuxThreads, 0, stream, p, -1);
    }
    prof_end(2, stream);
    if (e != cudaSuccess) set_error("bwd_pre launch", e);
    return e;
}

// The item schedule of a launch (see BwdSched), kept for the last shape this
// host thread launched.  Items are numbered longest first, so list scheduling
// takes them in index order.
const BwdSched& item_schedule(int n_items, int BH, int n_qt, bool causal, int n_cta) {
    thread_local BwdSched sc;
    thread_local int key[5] = {-1, -1, -1, -1, -1};
    const int k[5] = {n_items, BH, n_qt, causal ? 1 : 0, n_cta};
    if (std::equal(k, k + 5, key)) return sc;
    std::copy(k, k + 5, key);
    sc.n = 0;
    if (n_items > kSchedMaxItems || n_cta > kSchedMaxCta || n_cta < 1) return sc;
    std::vector<std::vector<int>> per(static_cast<size_t>(n_cta));
    using Slot = std::pair<long long, int>;  // (query tiles so far, CTA)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> least;
    for (int c = 0; c < n_cta; ++c) least.push({0, c});
    for (int it = 0; it < n_items; ++it) {
        const int kt = it / BH;
        const int tiles = causal ? n_qt - kt : n_qt;
        const Slot s0 = least.top();
        least.pop();
        per[static_cast<size_t>(s0.second)].push_back(it);
        least.push({s0.first + tiles, s0.second});
    }
    int pos = 0;
    for (int c = 0; c < n_cta; ++c) {
        sc.start[c] = static_cast<uint16_t>(pos);
        for (int it : per[static_cast<size_t>(c)]) sc.items[pos++] = static_cast<uint16_t>(it);
    }
    sc.start[n_cta] = static_cast<uint16_t>(pos);
    sc.n = pos;
    return sc;
}

template <int D, bool CAUSAL>
cudaError_t launch_main(const BwdArgs& a, const BwdParams& p, cudaStream_t stream) {
    using L = BwdLayout<D>;
    auto kern = bwd_kernel<D, CAUSAL>;
    static unsigned smem_set = 0;  // devices on which this instantiation's limit is raised
    cudaError_t e = smem_limit_once(kern, L::kAlloc, &smem_set);
    if (e != cudaSuccess) {
        set_error("bwd_main cudaFuncSetAttribute", e);
        return e;
    }
    // persistent: one CTA per SM (or per item, if fewer)
    const int n_cta = p.n_items < a.num_sms ? p.n_items : a.num_sms;
    prof_begin(3, stream);
    const BwdSched& sched = item_schedule(p.n_items, p.BH, (p.N + kBlockM - 1) / kBlockM, CAUSAL, n_cta);
    e = launch_pdl(kern, dim3(static_cast<unsigned>(n_cta > 0 ? n_cta : 1)), L::kThreads, L::kAlloc, stream,
                   *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dqacc, *a.tm_dk, *a.tm_dv, p, sched);
    prof_end(3, stream);
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

template <int D>
cudaError_t launch_convert(const BwdParams& p, int num_sms, cudaStream_t stream) {
    prof_begin(4, stream);
    const cudaError_t e = launch_pdl(dq_convert_kernel<D>, dim3(static_cast<unsigned>(num_sms * kAuxBlocksPerSM)),
                                     kAuxThreads, 0, stream, p);
    prof_end(4, stream);
    if (e != cudaSuccess) set_error("dq_convert launch", e);
    return e;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
    const BwdParams p = make_params(a);
    cudaError_t e;
    if (a.d == 64) {
        if ((e = launch_pre<64>(p, a.num_sms, stream)) != cudaSuccess) return e;
        e = a.causal ? launch_main<64, true>(a, p, stream) : launch_main<64, false>(a, p, stream);
        if (e != cudaSuccess) return e;
        return launch_convert<64>(p, a.num_sms, stream);
    }
    if ((e = launch_pre<128>(p, a.num_sms, stream)) != cudaSuccess) return e;
    e = a.causal ? launch_main<128, true>(a, p, stream) : launch_main<128, false>(a, p, stream);
    if (e != cudaSuccess) return e;
    return launch_convert<128>(p, a.num_sms, stream);
}

}  // namespace fa
