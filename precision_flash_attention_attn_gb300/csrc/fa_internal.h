// Internal launch interface shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kBlockM = 128;  // query rows per tile (one TMEM lane per row)
constexpr int kBlockN = 128;  // keys per tile

// Where row n of head bh = b*H + h of a [*, N, d] tensor (q, k, v, o, dO,
// dq, dk, dv) starts, in elements: b*sB + h*sH + n*sN; the d elements of a
// row are contiguous.  [B, H, N, d]: sN = d, sH = N*d, sB = H*N*d;
// [B, N, H, d]: sN = H*d, sH = d, sB = N*H*d.
// The tensor maps list the dimensions in increasing stride order: (d, N, H,
// B) for [B, H, N, d] and (d, H, N, B) for [B, N, H, d] (head_inner = 1), so
// a tile's coordinates are (column, row, head, batch) or (column, head, row,
// batch).
struct RowLayout {
    int H;
    int head_inner;
    long long sN, sH, sB;
    __host__ __device__ size_t row(int bh, int n) const {
        return static_cast<size_t>(bh / H) * static_cast<size_t>(sB) +
               static_cast<size_t>(bh % H) * static_cast<size_t>(sH) + static_cast<size_t>(n) * static_cast<size_t>(sN);
    }
};


struct FwdArgs {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    const CUtensorMap* tm_o;  // O as a TMA store target (the statistics variant ignores it)
    void* o;            // [BH, N, d] BF16 (modes 0, 1) or FP32 (mode 2); null: not written
    float* lse;         // [BH, N]; null: not written
    int32_t* tie_count; // statistics variant only: [BH, N]
    int32_t* p_one;     // statistics variant only, nullable: [2][BH, N]
    int BH, N, d, causal, mode;
    float scale;        // alpha
    float scale_log2;   // alpha * log2(e)
    float beta;         // stabilised-softmax shift factor (mode 1)
    int* status;        // device status word
    int num_sms;        // persistent grid: at most one CTA per SM
    int test_withhold_k;  // test hook: CTA 0 skips its first K tile load, so
                          // the waits on it time out (FA_TEST_WITHHOLD_K=1)
    const float* shift;   // nullable, mode 1: fixed per-row shift [BH, N] (raw
                          // score units) used from the first key tile on
    const int32_t* rs_in; // nullable, statistics variant: tie counts to report
    uint64_t head_mask = ~0ull;  // heads h (bit h, h < 64) computed by this launch; ~0: all
    int H = 0;                   // heads per batch (for head_mask)
    RowLayout lay;               // q, k, v, o (the maps are built with the same strides)
};

// Row statistics pre-pass of the stabilised softmax with a tolerance eps:
// per row the maximum rm of the raw scores, rs = #{j: scale*(rm - s_j) <= eps}
// and the mode's shift m(rm, rs).
struct RowShiftArgs {
    const void* q;
    const void* k;
    float* shift;   // nullable: [BH, N] shift, raw score units
    int32_t* rs;    // nullable: [BH, N] near-tie counts
    int BH, N, d, causal, mode;
    float scale, beta, eps;
    RowLayout lay;  // q, k
};
cudaError_t launch_row_shift(const RowShiftArgs& a, cudaStream_t stream);

// delta = rowsum(dP o P) pre-pass of the backward (written as -scale*delta
// into the padded row array [BH, Npad]).
struct DeltaPdpArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* dout;
    const float* lse;  // [BH, N]
    float* delta;      // [BH, Npad]
    int BH, N, Npad, d, causal;
    float scale;
};
cudaError_t launch_delta_pdp(const DeltaPdpArgs& a, cudaStream_t stream);

struct BwdArgs {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    const CUtensorMap* tm_do;
    const CUtensorMap* tm_dqacc;  // FP32 [BH, N, d] accumulator (reduce-add target)
    const CUtensorMap* tm_dk;     // dK, dV as TMA store targets (BF16 [BH, N, d], 64 x 32 boxes)
    const CUtensorMap* tm_dv;
    const void* o;                // [BH, N, d] BF16 or FP32 (mode 2)
    const float* lse;             // [BH, N]
    const void* dout;             // [BH, N, d] BF16
    float* dq_acc;                // FP32 [BH, N, d] workspace
    float* lse2;                  // FP32 [BH, Npad] workspace: LSE * log2(e)
    float* delta;                 // FP32 [BH, Npad] workspace: rowsum(dO o O)
    int zero_acc;                 // 1: the pre kernel clears dq_acc
    int delta_given;              // 1: delta is already in place (rowsum(dP o P) pre-pass)
    const float* o32 = nullptr;   // per-head modes: FP32 O of the heads in fp32_mask
    uint64_t fp32_mask = 0;       // heads h (bit h) whose delta uses o32 instead of o
    int H = 0;
    RowLayout lay;                // q, k, v, o, dO, dq, dk, dv (dq_acc is [BH, N, d])
    void* dq;                     // [BH, N, d] BF16
    void* dk;
    void* dv;
    int BH, N, Npad, d, causal, mode;
    float scale, scale_log2;
    int* status;
    int num_sms;
};

// Record the CUDA error behind a failing step (read back by fa_last_error).
void set_error(const char* step, cudaError_t e);
void set_error_msg(const char* step, const char* msg);

// Kernel timing hooks (no-ops unless a profiling session is active).
void prof_begin(int kind, cudaStream_t stream);
void prof_end(int kind, cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit the first time it launches on
// each device (the setting belongs to the function on that device and stays;
// repeating the call on every launch only costs host time).  `done` is a
// per-kernel bit mask of devices already set.
template <typename Kernel>
inline cudaError_t smem_limit_once(Kernel kern, int bytes, unsigned* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned bit = (dev >= 0 && dev < 32) ? (1u << dev) : 0u;
    if (bit && (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) __atomic_fetch_or(done, bit, __ATOMIC_RELEASE);
    return e;
}

cudaError_t launch_fwd(const FwdArgs& a, bool stats, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);

}  // namespace fa
