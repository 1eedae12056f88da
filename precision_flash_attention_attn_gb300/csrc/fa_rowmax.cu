// Row pre-passes on CUDA cores.
//
// Row maximum and near-tie count of the raw scores, the two row statistics of
// the stabilised safe softmax ("Why Low-Precision Transformer Training Fails:
// An Analysis on Flash Attention", section 3.4.5, "The modified safe
// softmax"):
//   rm = max_j q.k_j,   rs = #{ j : scale * (rm - q.k_j) <= eps }
// over the visible keys, and the shift of the mode: m = beta*rm if rm > 0 and
// rs > 1, 0 if rm < 0 and rs > 1, rm otherwise (mode 1), rm (modes 0, 2).
// With eps > 0 a key's membership depends on the row's final maximum, which a
// single tiled pass does not know while it exponentiates, so the forward takes
// the shift from this pre-pass instead of from its running state.
//
// One CTA = 128 query rows of one (batch, head), one thread per row, FP32
// scores on CUDA cores with one fixed FMA order, so both passes see the same
// values.  Keys are staged 32 at a time in shared memory as FP32.
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {
namespace {

__device__ __forceinline__ float bf16_load(const void* base, size_t idx) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

template <int D>
__global__ void __launch_bounds__(128) row_shift_kernel(const RowShiftArgs a) {
    constexpr int KC = 32;
    __shared__ float sk[KC][D + 1];
    const int bh = blockIdx.y;
    const int r0 = blockIdx.x * 128;
    const int i = r0 + threadIdx.x;
    const bool valid = i < a.N;
    float q[D];
#pragma unroll
    for (int c = 0; c < D; ++c) q[c] = valid ? bf16_load(a.q, a.lay.row(bh, i) + c) : 0.f;
    const int kend = a.causal ? min(a.N, r0 + 128) : a.N;
    auto load_k = [&](int j0) {
        for (int e = threadIdx.x; e < KC * D; e += 128) {
            const int jj = e / D, c = e % D;
            const int j = j0 + jj;
            sk[jj][c] = (j < kend) ? bf16_load(a.k, a.lay.row(bh, j) + c) : 0.f;
        }
    };
    auto score = [&](int jj) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) s = fmaf(q[c], sk[jj][c], s);
        return s;
    };
    auto visible = [&](int j) { return j < kend && (!a.causal || j <= i); };

    float rm = -INFINITY;
    for (int j0 = 0; j0 < kend; j0 += KC) {
        __syncthreads();
        load_k(j0);
        __syncthreads();
        for (int jj = 0; jj < KC; ++jj)
            if (visible(j0 + jj)) rm = fmaxf(rm, score(jj));
    }
    int rs = 0;
    for (int j0 = 0; j0 < kend; j0 += KC) {
        __syncthreads();
        load_k(j0);
        __syncthreads();
        for (int jj = 0; jj < KC; ++jj) {
            if (!visible(j0 + jj)) continue;
            const float s = score(jj);
            rs += (a.eps == 0.f) ? (s == rm ? 1 : 0) : (a.scale * (rm - s) <= a.eps ? 1 : 0);
        }
    }
    if (!valid) return;
    float m = rm;
    if (a.mode == 1 && rs > 1) {
        if (rm > 0.f) m = a.beta * rm;
        else if (rm < 0.f) m = 0.f;
    }
    const size_t row = static_cast<size_t>(bh) * a.N + i;
    if (a.shift) a.shift[row] = m;
    if (a.rs) a.rs[row] = rs;
}

// delta = rowsum(dP o P) of the backward, with P = exp(scale * q.k - LSE)
// recomputed from the saved LSE and dP = dO . v, both in FP32 over the visible
// keys, summed with a compensated (Kahan) sum: in exact arithmetic this equals
// rowsum(dO o O) for the exact O, without the stored output's rounding
// (section 3.4.2, "Failure is linked to the computation of delta"; the delta
// substitution experiment of section 5).  Written pre-negated and pre-scaled
// (-scale * delta) into the backward's padded row array [BH, Npad]; padded
// rows get 0.
template <int D>
__global__ void __launch_bounds__(128) delta_pdp_kernel(const DeltaPdpArgs a) {
    constexpr int KC = 32;
    __shared__ float sk[KC][D + 1];
    __shared__ float sv[KC][D + 1];
    const int bh = blockIdx.y;
    const int r0 = blockIdx.x * 128;
    const int i = r0 + threadIdx.x;
    const bool valid = i < a.N;
    const size_t head = static_cast<size_t>(bh) * a.N * D;

    float q[D], g[D];
#pragma unroll
    for (int c = 0; c < D; ++c) {
        q[c] = valid ? bf16_load(a.q, head + static_cast<size_t>(i) * D + c) : 0.f;
        g[c] = valid ? bf16_load(a.dout, head + static_cast<size_t>(i) * D + c) : 0.f;
    }
    const float lse = valid ? a.lse[static_cast<size_t>(bh) * a.N + i] : 0.f;
    const int kend = a.causal ? min(a.N, r0 + 128) : a.N;
    float acc = 0.f, comp = 0.f;
    for (int j0 = 0; j0 < kend; j0 += KC) {
        __syncthreads();
        for (int e = threadIdx.x; e < KC * D; e += 128) {
            const int jj = e / D, c = e % D;
            const int j = j0 + jj;
            const bool in = j < kend;
            sk[jj][c] = in ? bf16_load(a.k, head + static_cast<size_t>(j) * D + c) : 0.f;
            sv[jj][c] = in ? bf16_load(a.v, head + static_cast<size_t>(j) * D + c) : 0.f;
        }
        __syncthreads();
        for (int jj = 0; jj < KC; ++jj) {
            const int j = j0 + jj;
            if (j >= kend || (a.causal && j > i)) continue;
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) {
                s = fmaf(q[c], sk[jj][c], s);
                dp = fmaf(g[c], sv[jj][c], dp);
            }
            const float y = expf(fmaf(a.scale, s, -lse)) * dp - comp;
            const float t = acc + y;
            comp = (t - acc) - y;
            acc = t;
        }
    }
    const size_t row = static_cast<size_t>(bh) * a.Npad + i;
    if (i < a.Npad) a.delta[row] = valid ? -a.scale * acc : 0.f;
}

}  // namespace

cudaError_t launch_delta_pdp(const DeltaPdpArgs& a, cudaStream_t stream) {
    // every padded row of every head is written (0 past N)
    dim3 grid(static_cast<unsigned>(a.Npad / 128), static_cast<unsigned>(a.BH));
    if (a.d == 64)
        delta_pdp_kernel<64><<<grid, 128, 0, stream>>>(a);
    else
        delta_pdp_kernel<128><<<grid, 128, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) set_error("delta_pdp launch", e);
    return e;
}

cudaError_t launch_row_shift(const RowShiftArgs& a, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>((a.N + 127) / 128), static_cast<unsigned>(a.BH));
    if (a.d == 64)
        row_shift_kernel<64><<<grid, 128, 0, stream>>>(a);
    else
        row_shift_kernel<128><<<grid, 128, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) set_error("row_shift launch", e);
    return e;
}

}  // namespace fa
