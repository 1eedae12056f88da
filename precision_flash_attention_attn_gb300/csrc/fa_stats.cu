// Signed rounding error of the stored attention output, per row:
//   pv_err[r] = sum_c (o[r,c] - O_ref[r,c])
// where O_ref = softmax(scale * q_r K^T) V is recomputed on CUDA cores in FP32
// with the exact row maximum and compensated (Kahan) sums, independently of
// the tensor-core forward ("Why Low-Precision Transformer Training Fails: An
// Analysis on Flash Attention", section 3.4.4, "Isolating the error to PV":
// the low-precision result minus the FP32 result).  Optionally also the error
// of the backward's delta = rowsum(dO o O) that the stored output causes,
//   delta_err[r] = sum_c dO[r,c] * (o[r,c] - O_ref[r,c])  (= delta_lp - delta_hp,
// section 3.4.4 "Cause 2", with O_ref standing in for O_hp).  Diagnostic only.
//
// One CTA = 128 query rows of one (batch, head), one thread per row.  Keys are
// staged 32 at a time in shared memory as FP32.  Pass 1 finds the row max;
// then one pass per 32-column slice accumulates sum_j p_j v_j[slice] (and, in
// the first slice, l = sum_j p_j).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_stats.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

struct Kahan {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
};

__device__ __forceinline__ float bf16_at(const void* base, size_t idx) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

template <int D>
__global__ void __launch_bounds__(128) pv_err_kernel(const StatsArgs a) {
    constexpr int KC = 32;
    __shared__ float sk[KC][D + 1];
    __shared__ float sv[KC][KC + 1];
    const int bh = blockIdx.y;
    const int r0 = blockIdx.x * 128;
    const int i = r0 + threadIdx.x;
    const bool valid = i < a.N;
    const size_t head = static_cast<size_t>(bh) * a.N * D;

    float q[D];
#pragma unroll
    for (int c = 0; c < D; ++c) q[c] = valid ? bf16_at(a.q, head + static_cast<size_t>(i) * D + c) : 0.f;
    const int kend = a.causal ? min(a.N, r0 + 128) : a.N;

    auto load_k = [&](int j0) {
        for (int e = threadIdx.x; e < KC * D; e += 128) {
            const int jj = e / D, c = e % D;
            const int j = j0 + jj;
            sk[jj][c] = (j < kend) ? bf16_at(a.k, head + static_cast<size_t>(j) * D + c) : 0.f;
        }
    };
    auto score = [&](int jj) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) s = fmaf(q[c], sk[jj][c], s);
        return s;
    };
    auto visible = [&](int j) { return j < kend && (!a.causal || j <= i); };

    float mx = -INFINITY;
    for (int j0 = 0; j0 < kend; j0 += KC) {
        __syncthreads();
        load_k(j0);
        __syncthreads();
        for (int jj = 0; jj < KC; ++jj)
            if (visible(j0 + jj)) mx = fmaxf(mx, score(jj));
    }

    Kahan l;
    Kahan err;
    Kahan derr;
    for (int c0 = 0; c0 < D; c0 += KC) {
        Kahan acc[KC];
        for (int j0 = 0; j0 < kend; j0 += KC) {
            __syncthreads();
            load_k(j0);
            for (int e = threadIdx.x; e < KC * KC; e += 128) {
                const int jj = e / KC, c = e % KC;
                const int j = j0 + jj;
                sv[jj][c] = (j < kend) ? bf16_at(a.v, head + static_cast<size_t>(j) * D + c0 + c) : 0.f;
            }
            __syncthreads();
            for (int jj = 0; jj < KC; ++jj) {
                if (!visible(j0 + jj)) continue;
                const float pj = expf(a.scale * (score(jj) - mx));
                if (c0 == 0) l.add(pj);
#pragma unroll
                for (int c = 0; c < KC; ++c) acc[c].add(pj * sv[jj][c]);
            }
        }
        if (valid) {
            const float inv = 1.f / l.s;
#pragma unroll
            for (int c = 0; c < KC; ++c) {
                const size_t idx = head + static_cast<size_t>(i) * D + c0 + c;
                const float oc = (a.mode == 2) ? static_cast<const float*>(a.o)[idx] : bf16_at(a.o, idx);
                const float e = oc - acc[c].s * inv;
                err.add(e);
                if (a.delta_err) derr.add(bf16_at(a.dout, idx) * e);
            }
        }
    }
    if (valid) {
        a.pv_err[static_cast<size_t>(bh) * a.N + i] = err.s;
        if (a.delta_err) a.delta_err[static_cast<size_t>(bh) * a.N + i] = derr.s;
    }
}

// The decomposition of delta_lp - delta_hp for a stored output o (section
// 3.4.4, "Cause 2"; the quantitative decomposition the page lists as
// missing), per row, in FP32 on CUDA cores:
//   P_j = exp(scale*s_j - m) with the row's shift m (the untiled rule of the
//   mode, tolerance eps), b_j = bf16(P_j), l = sum_j P_j, p_j = the FP32
//   reference probabilities (exact row maximum, compensated sums);
//   one  = sum_c dO[c] sum_{j: b_j = 1}  (b_j / l - p_j) v_j[c]
//   rest = sum_c dO[c] sum_{j: b_j != 1} (b_j / l - p_j) v_j[c]
//   out  = sum_c dO[c] (o[c] - sum_j b_j v_j[c] / l)
// One thread per row, keys staged 32 at a time, 8 output columns per pass.
template <int D>
__global__ void __launch_bounds__(128) delta_split_kernel(const SplitArgs a) {
    constexpr int KC = 32;
    constexpr int CW = 8;
    __shared__ float sk[KC][D + 1];
    __shared__ float sv[KC][CW + 1];
    const int bh = blockIdx.y;
    const int r0 = blockIdx.x * 128;
    const int i = r0 + threadIdx.x;
    const bool valid = i < a.N;
    const size_t head = static_cast<size_t>(bh) * a.N * D;

    float q[D];
#pragma unroll
    for (int c = 0; c < D; ++c) q[c] = valid ? bf16_at(a.q, head + static_cast<size_t>(i) * D + c) : 0.f;
    const int kend = a.causal ? min(a.N, r0 + 128) : a.N;
    auto load_k = [&](int j0) {
        for (int e = threadIdx.x; e < KC * D; e += 128) {
            const int jj = e / D, c = e % D;
            const int j = j0 + jj;
            sk[jj][c] = (j < kend) ? bf16_at(a.k, head + static_cast<size_t>(j) * D + c) : 0.f;
        }
    };
    auto score = [&](int jj) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) s = fmaf(q[c], sk[jj][c], s);
        return s;
    };
    auto visible = [&](int j) { return j < kend && (!a.causal || j <= i); };

    // the row's maximum, (near-)tie count and shift
    float rm = -INFINITY;
    for (int j0 = 0; j0 < kend; j0 += KC) {
        __syncthreads();
        load_k(j0);
        __syncthreads();
        for (int jj = 0; jj < KC; ++jj)
            if (visible(j0 + jj)) rm = fmaxf(rm, score(jj));
    }
    int rs = 0;
    Kahan lref, l;
    float m = 0.f;
    for (int pass = 0; pass < 2; ++pass) {
        for (int j0 = 0; j0 < kend; j0 += KC) {
            __syncthreads();
            load_k(j0);
            __syncthreads();
            for (int jj = 0; jj < KC; ++jj) {
                if (!visible(j0 + jj)) continue;
                const float sc = score(jj);
                if (pass == 0) {
                    rs += (a.eps == 0.f) ? (sc == rm ? 1 : 0) : (a.scale * (rm - sc) <= a.eps ? 1 : 0);
                } else {
                    lref.add(expf(a.scale * (sc - rm)));
                    l.add(expf(a.scale * (sc - m)));
                }
            }
        }
        if (pass == 0) {
            m = rm;
            if (a.mode == 1 && rs > 1) {
                if (rm > 0.f) m = a.beta * rm;
                else if (rm < 0.f) m = 0.f;
            }
        }
    }
    float e_one = 0.f, e_rest = 0.f, e_out = 0.f;
    for (int c0 = 0; c0 < D; c0 += CW) {
        Kahan b1[CW], p1[CW], b2[CW], p2[CW];
        for (int j0 = 0; j0 < kend; j0 += KC) {
            __syncthreads();
            load_k(j0);
            for (int e = threadIdx.x; e < KC * CW; e += 128) {
                const int jj = e / CW, c = e % CW;
                const int j = j0 + jj;
                sv[jj][c] = (j < kend) ? bf16_at(a.v, head + static_cast<size_t>(j) * D + c0 + c) : 0.f;
            }
            __syncthreads();
            for (int jj = 0; jj < KC; ++jj) {
                if (!visible(j0 + jj)) continue;
                const float sc = score(jj);
                const float pb = __bfloat162float(__float2bfloat16_rn(expf(a.scale * (sc - m))));
                const float pr = expf(a.scale * (sc - rm)) / lref.s;
#pragma unroll
                for (int c = 0; c < CW; ++c) {
                    if (pb == 1.f) {
                        b1[c].add(pb * sv[jj][c]);
                        p1[c].add(pr * sv[jj][c]);
                    } else {
                        b2[c].add(pb * sv[jj][c]);
                        p2[c].add(pr * sv[jj][c]);
                    }
                }
            }
        }
        if (valid) {
#pragma unroll
            for (int c = 0; c < CW; ++c) {
                const size_t idx = head + static_cast<size_t>(i) * D + c0 + c;
                const float g = bf16_at(a.dout, idx);
                const float oc = (a.mode == 2) ? static_cast<const float*>(a.o)[idx] : bf16_at(a.o, idx);
                e_one += g * (b1[c].s / l.s - p1[c].s);
                e_rest += g * (b2[c].s / l.s - p2[c].s);
                e_out += g * (oc - (b1[c].s + b2[c].s) / l.s);
            }
        }
    }
    if (valid) {
        const size_t row = static_cast<size_t>(bh) * a.N + i;
        a.err_one[row] = e_one;
        a.err_rest[row] = e_rest;
        a.err_out[row] = e_out;
    }
}

}  // namespace

cudaError_t launch_delta_split(const SplitArgs& a, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>((a.N + 127) / 128), static_cast<unsigned>(a.BH));
    if (a.d == 64)
        delta_split_kernel<64><<<grid, 128, 0, stream>>>(a);
    else
        delta_split_kernel<128><<<grid, 128, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) set_error("delta_split launch", e);
    return e;
}

cudaError_t launch_pv_err(const StatsArgs& a, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>((a.N + 127) / 128), static_cast<unsigned>(a.BH));
    prof_begin(5, stream);
    if (a.d == 64)
        pv_err_kernel<64><<<grid, 128, 0, stream>>>(a);
    else
        pv_err_kernel<128><<<grid, 128, 0, stream>>>(a);
    prof_end(5, stream);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) set_error("pv_err launch", e);
    return e;
}

}  // namespace fa
