// C ABI of libfa (declared in include/fa.h): argument validation, device
// checks, TMA tensor-map construction, workspace handling and dispatch to the
// kernels.  No torch types, no exceptions across the boundary.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "fa_stats.h"

namespace {

// Device word where kernels record bounded-wait timeouts (one per device; the
// host reaches it through its device address).
__device__ int g_fa_status;

constexpr int kMaxDevices = 64;

thread_local char g_last_error[256];

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int* status = nullptr;
    int num_sms = 0;
    int dev = 0;
    uint64_t pool_threshold = 0;  // release threshold this library has set on the device's mempool
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(const char* step, cudaError_t e) {
    fa::set_error(step, e);
    return FA_ERR_CUDA;
}

// Current device: sm_103 check and the status word address.
int device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail("cudaGetDevice", ce);
    if (dev < 0 || dev >= kMaxDevices) {
        fa::set_error_msg("device_info", "device index exceeds the library's device table (64)");
        return FA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.probed) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        di.supported = (major == 10 && minor == 3);
        if (di.supported &&
            cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        if (di.supported) {
            void* p = nullptr;
            ce = cudaGetSymbolAddress(&p, g_fa_status);
            if (ce != cudaSuccess) return cuda_fail("cudaGetSymbolAddress(status word)", ce);
            di.status = static_cast<int*>(p);
        }
        di.dev = dev;
        di.probed = true;
    }
    if (!di.supported) return FA_ERR_UNSUPPORTED;
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return FA_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = &di;
    return FA_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int N, int d, int causal, float scale, int mode) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (mode < 0 || mode > 2) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    const long long total = static_cast<long long>(B) * H * N * (d > 0 ? d : 1);
    if (total >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    if (N > 65535 * fa::kBlockM) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// 3-D view [BH][N][d] of a row-major tensor; box = inner x rows x 1,
// 128-byte swizzle (inner * elem_bytes == 128).
int make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int BH, int N, int d,
             int inner, int rows = fa::kBlockM) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                             static_cast<cuuint64_t>(d) * N * elem_bytes};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[64];
        snprintf(msg, sizeof msg, "CUresult %d", static_cast<int>(r));
        fa::set_error_msg("cuTensorMapEncodeTiled", msg);
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

// Row strides of the [*, N, d] tensors in a layout (FA_LAYOUT_*).
fa::RowLayout layout_of(int layout, int H, int N, int d) {
    fa::RowLayout l{};
    l.H = H;
    if (layout == FA_LAYOUT_BNHD) {
        l.head_inner = 1;
        l.sN = static_cast<long long>(H) * d;
        l.sH = d;
        l.sB = static_cast<long long>(N) * H * d;
    } else {
        l.head_inner = 0;
        l.sN = d;
        l.sH = static_cast<long long>(N) * d;
        l.sB = static_cast<long long>(H) * N * d;
    }
    return l;
}

// 4-D view of a [*, N, d] tensor in layout `lay`, dimensions in increasing
// stride order (see fa::RowLayout); box = inner x rows (x 1 head x 1 batch),
// 128-byte swizzle (inner * elem_bytes == 128).
int make_rows_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, const fa::RowLayout& lay,
                  int B, int N, int d, int inner, int rows = fa::kBlockM) {
    const cuuint64_t e = static_cast<cuuint64_t>(elem_bytes);
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    dims[0] = static_cast<cuuint64_t>(d);
    dims[3] = static_cast<cuuint64_t>(B);
    strides[2] = static_cast<cuuint64_t>(lay.sB) * e;
    box[0] = static_cast<cuuint32_t>(inner);
    box[3] = 1;
    if (lay.head_inner) {
        dims[1] = static_cast<cuuint64_t>(lay.H);
        dims[2] = static_cast<cuuint64_t>(N);
        strides[0] = static_cast<cuuint64_t>(lay.sH) * e;
        strides[1] = static_cast<cuuint64_t>(lay.sN) * e;
        box[1] = 1;
        box[2] = static_cast<cuuint32_t>(rows);
    } else {
        dims[1] = static_cast<cuuint64_t>(N);
        dims[2] = static_cast<cuuint64_t>(lay.H);
        strides[0] = static_cast<cuuint64_t>(lay.sN) * e;
        strides[1] = static_cast<cuuint64_t>(lay.sH) * e;
        box[1] = static_cast<cuuint32_t>(rows);
        box[2] = 1;
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[64];
        snprintf(msg, sizeof msg, "CUresult %d", static_cast<int>(r));
        fa::set_error_msg("cuTensorMapEncodeTiled", msg);
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

// Stabilised-softmax parameters (NULL: the defaults).  "The modified safe
// softmax" of section 3.4.5 requires beta > 1 and a tolerance eps >= 0.
int check_params(const fa_stab_params_t* prm, float* beta, float* eps) {
    *beta = FA_STAB_BETA_DEFAULT;
    *eps = 0.f;
    if (!prm) return FA_OK;
    if (!std::isfinite(prm->beta) || !(prm->beta > 1.f)) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(prm->eps) || prm->eps < 0.f) return FA_ERR_INVALID_ARG;
    *beta = prm->beta;
    *eps = prm->eps;
    return FA_OK;
}

// Enqueue the row pre-pass (row maximum, near-tie count, shift).
int launch_row_pass(const void* q, const void* k, int BH, int N, int d, int causal, float scale, int mode,
                    float beta, float eps, float* shift, int32_t* rs, cudaStream_t st, const fa::RowLayout& lay) {
    fa::RowShiftArgs r{};
    r.lay = lay;
    r.q = q;
    r.k = k;
    r.shift = shift;
    r.rs = rs;
    r.BH = BH;
    r.N = N;
    r.d = d;
    r.causal = causal;
    r.mode = mode;
    r.scale = scale;
    r.beta = beta;
    r.eps = eps;
    return fa::launch_row_shift(r, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

float log2e_times(float scale) { return static_cast<float>(static_cast<double>(scale) * 1.4426950408889634); }

// Backward workspace, two regions:
//   zero region  [FP32 dQ accumulator BH*N*d]: zero when the main kernel
//                starts; a fresh workspace is cleared by the pre kernel, the
//                allocation-free one is left zeroed by the previous call's
//                conversion;
//   row region   [-LSE*log2e BH*Npad][-alpha*delta BH*Npad]: written by the
//                pre kernel.
// Both start on a 256-byte boundary (BH*N*d*4 is a multiple of 256).
struct BwdSizes {
    size_t acc, rows;  // accumulator, one of the two row arrays
    size_t zero_bytes() const { return acc; }
    size_t row_bytes() const { return 2 * rows; }
};

BwdSizes bwd_sizes(int BH, int N, int d) {
    const int n_qt = (N + fa::kBlockM - 1) / fa::kBlockM;
    BwdSizes z;
    z.acc = static_cast<size_t>(BH) * N * d * sizeof(float);
    z.rows = static_cast<size_t>(BH) * n_qt * fa::kBlockM * sizeof(float);
    return z;
}

bool bwd_pointers_ok(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     const void* dq, const void* dk, const void* dv) {
    return aligned16(q) && aligned16(k) && aligned16(v) && aligned16(o) && aligned16(lse) && aligned16(dO) &&
           aligned16(dq) && aligned16(dk) && aligned16(dv);
}

// Enqueue the backward kernels.  `zero` is the zero region (bwd_sizes
// layout), which the first kernel clears right before the main kernel adds
// into it (its lines are then still in L2), `rows` the row region.
// Arguments are already validated.
int launch_backward(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                    void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, int mode,
                    const DeviceInfo* di, void* zero, void* rows, cudaStream_t st, int delta_given = 0,
                    const float* o32 = nullptr, uint64_t fp32_mask = 0, int layout = FA_LAYOUT_BHND) {
    const int BH = B * H;
    const fa::RowLayout lay = layout_of(layout, H, N, d);
    const int Npad = (N + fa::kBlockM - 1) / fa::kBlockM * fa::kBlockM;
    char* zb = static_cast<char*>(zero);
    float* dq_acc = reinterpret_cast<float*>(zb);
    float* lse2 = static_cast<float*>(rows);
    float* delta = lse2 + static_cast<size_t>(BH) * Npad;
    CUtensorMap mq, mk, mv, mdo, macc, mdk, mdv;
    if (make_rows_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mdo, dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_map(&macc, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BH, N, d, 32, 32) ||
        make_rows_map(&mdk, dk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64, 32) ||
        make_rows_map(&mdv, dv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64, 32))
        return FA_ERR_CUDA;
    fa::BwdArgs a{};
    a.tm_q = &mq;
    a.tm_k = &mk;
    a.tm_v = &mv;
    a.tm_do = &mdo;
    a.tm_dqacc = &macc;
    a.tm_dk = &mdk;
    a.tm_dv = &mdv;
    a.o = o;
    a.lse = lse;
    a.dout = dO;
    a.dq_acc = dq_acc;
    a.lse2 = lse2;
    a.delta = delta;
    a.zero_acc = 1;
    a.delta_given = delta_given;
    a.o32 = o32;
    a.fp32_mask = fp32_mask;
    a.H = H;
    a.lay = lay;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.BH = BH;
    a.N = N;
    a.Npad = Npad;
    a.d = d;
    a.causal = causal;
    a.mode = mode;
    a.scale = scale;
    a.scale_log2 = log2e_times(scale);
    a.status = di->status;
    a.num_sms = di->num_sms;
    return fa::launch_bwd(a, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Keep at least `bytes` of the current device's stream-ordered pool reserved
// across synchronisations, so that steady-state workspace allocations are
// served from the pool instead of the OS.  Only ever raises the threshold.
void reserve_pool(DeviceInfo* di, size_t bytes) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (di->pool_threshold >= bytes) return;
    cudaMemPool_t pool;
    if (cudaDeviceGetMemPool(&pool, di->dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    cuuint64_t cur = 0;
    if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &cur) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    if (cur < bytes) {
        cuuint64_t want = bytes;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &want) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        cur = want;
    }
    di->pool_threshold = cur;
}

}  // namespace

namespace fa {

void set_error_msg(const char* step, const char* msg) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", step, msg);
}

void set_error(const char* step, cudaError_t e) { set_error_msg(step, cudaGetErrorString(e)); }

}  // namespace fa

extern "C" {

const char* fa_last_error(void) { return g_last_error; }

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_ALLOC: return "FA_ERR_ALLOC";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        case FA_ERR_NONFINITE: return "FA_ERR_NONFINITE";
        default: return "FA_ERR_UNKNOWN";
    }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           int causal, float scale, int mode, fa_stream_t stream) {
    return fa_fwd_ex(q, k, v, o, lse, B, H, N, d, causal, scale, mode, nullptr, stream);
}

}  // extern "C"

namespace {

// The forward of one mode over the heads in head_mask (~0: all), arguments
// already validated.
int run_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                int causal, float scale, int mode, float beta, float eps, uint64_t head_mask, const DeviceInfo* di,
                cudaStream_t st, int layout = FA_LAYOUT_BHND) {
    const int BH = B * H;
    const fa::RowLayout lay = layout_of(layout, H, N, d);
    CUtensorMap mq, mk, mv, mo;
    // O as a TMA store target: 64 BF16 or 32 FP32 columns (128 bytes) per box row
    const bool o32 = (mode == 2);
    if (make_rows_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mo, o, o32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o32 ? 4 : 2,
                      lay, B, N, d, o32 ? 32 : 64))
        return FA_ERR_CUDA;
    fa::FwdArgs a{};
    a.tm_q = &mq;
    a.tm_k = &mk;
    a.tm_v = &mv;
    a.tm_o = &mo;
    a.o = o;
    a.lse = lse;
    a.BH = BH;
    a.N = N;
    a.d = d;
    a.causal = causal;
    a.mode = mode;
    a.scale = scale;
    a.scale_log2 = log2e_times(scale);
    a.beta = beta;
    a.status = di->status;
    a.num_sms = di->num_sms;
    a.head_mask = head_mask;
    a.H = H;
    a.lay = lay;
    const char* hook = std::getenv("FA_TEST_WITHHOLD_K");
    a.test_withhold_k = (hook && hook[0] == '1') ? 1 : 0;
    if (mode != FA_MODE_STABILISED || eps == 0.f)
        return fa::launch_fwd(a, false, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    // A tolerance: each row's shift from a pre-pass over the whole row, held
    // fixed through the tiled forward (stream-ordered workspace, B*H*N*4 bytes).
    void* ws = nullptr;
    cudaError_t ae = cudaMallocAsync(&ws, static_cast<size_t>(BH) * N * sizeof(float), st);
    if (ae != cudaSuccess || !ws) {
        fa::set_error("cudaMallocAsync(row shifts)", ae);
        cudaGetLastError();
        return FA_ERR_ALLOC;
    }
    a.shift = static_cast<float*>(ws);
    int rc = launch_row_pass(q, k, BH, N, d, causal, scale, mode, beta, eps, static_cast<float*>(ws), nullptr, st, lay);
    if (rc == FA_OK && fa::launch_fwd(a, false, st) != cudaSuccess) rc = FA_ERR_CUDA;
    const cudaError_t fe = cudaFreeAsync(ws, st);
    if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(row shifts)", fe);
    return rc;
}

// Per-head modes: each of the H entries in {0, 1, 2}, H <= 64.  Sets the
// masks of the heads computed in each mode.
int check_head_modes(const int* head_modes, int H, uint64_t mask[3]) {
    mask[0] = mask[1] = mask[2] = 0;
    if (!head_modes) return FA_ERR_INVALID_ARG;
    if (H > 64) {
        fa::set_error_msg("per-head modes", "at most 64 heads per batch");
        return FA_ERR_UNSUPPORTED;
    }
    for (int h = 0; h < H; ++h) {
        if (head_modes[h] < 0 || head_modes[h] > 2) return FA_ERR_INVALID_ARG;
        mask[head_modes[h]] |= 1ull << h;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
              int causal, float scale, int mode, const fa_stab_params_t* params, fa_stream_t stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    float beta = 0.f, eps = 0.f;
    if ((rc = check_params(params, &beta, &eps))) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    return run_forward(q, k, v, o, lse, B, H, N, d, causal, scale, mode, beta, eps, ~0ull, di,
                       static_cast<cudaStream_t>(stream));
}

int fa_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  int causal, float scale, int mode, const fa_stab_params_t* params, int layout, fa_stream_t stream) {
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    float beta = 0.f, eps = 0.f;
    if ((rc = check_params(params, &beta, &eps))) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    return run_forward(q, k, v, o, lse, B, H, N, d, causal, scale, mode, beta, eps, ~0ull, di,
                       static_cast<cudaStream_t>(stream), layout);
}

int fa_fwd_heads(const void* q, const void* k, const void* v, void* o_bf16, float* o_fp32, float* lse, int B,
                 int H, int N, int d, int causal, float scale, const int* head_modes,
                 const fa_stab_params_t* params, fa_stream_t stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, 0);
    if (rc) return rc;
    uint64_t mask[3];
    if ((rc = check_head_modes(head_modes, H, mask))) return rc;
    if (((mask[0] | mask[1]) && !aligned16(o_bf16)) || (mask[2] && !aligned16(o_fp32))) return FA_ERR_INVALID_ARG;
    float beta = 0.f, eps = 0.f;
    if ((rc = check_params(params, &beta, &eps))) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int mode = 0; mode < 3 && rc == FA_OK; ++mode) {
        if (!mask[mode]) continue;
        void* o = (mode == 2) ? static_cast<void*>(o_fp32) : o_bf16;
        rc = run_forward(q, k, v, o, lse, B, H, N, d, causal, scale, mode, beta, eps, mask[mode], di, st);
    }
    return rc;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, int mode,
           fa_stream_t stream) {
    if (!bwd_pointers_ok(q, k, v, o, lse, dO, dq, dk, dv)) return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    const BwdSizes z = bwd_sizes(B * H, N, d);
    const size_t ws_bytes = z.zero_bytes() + z.row_bytes();
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const char* fail = std::getenv("FA_TEST_FAIL_ALLOC");
    if (fail && fail[0] == '1') return FA_ERR_ALLOC;
    reserve_pool(di, ws_bytes);
    void* ws = nullptr;
    cudaError_t ae = cudaMallocAsync(&ws, ws_bytes, st);
    if (ae != cudaSuccess || !ws) {
        fa::set_error("cudaMallocAsync(workspace)", ae);
        cudaGetLastError();
        return FA_ERR_ALLOC;
    }
    if (rc == FA_OK)
        rc = launch_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, di, ws,
                             static_cast<char*>(ws) + z.zero_bytes(), st);
    const cudaError_t fe = cudaFreeAsync(ws, st);
    if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(workspace)", fe);
    return rc;
}

int fa_bwd_layout(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, int mode,
                  int layout, fa_stream_t stream) {
    if (layout != FA_LAYOUT_BHND && layout != FA_LAYOUT_BNHD) return FA_ERR_INVALID_ARG;
    if (!bwd_pointers_ok(q, k, v, o, lse, dO, dq, dk, dv)) return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    const BwdSizes z = bwd_sizes(B * H, N, d);
    const size_t ws_bytes = z.zero_bytes() + z.row_bytes();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const char* fail = std::getenv("FA_TEST_FAIL_ALLOC");
    if (fail && fail[0] == '1') return FA_ERR_ALLOC;
    reserve_pool(di, ws_bytes);
    void* ws = nullptr;
    cudaError_t ae = cudaMallocAsync(&ws, ws_bytes, st);
    if (ae != cudaSuccess || !ws) {
        fa::set_error("cudaMallocAsync(workspace)", ae);
        cudaGetLastError();
        return FA_ERR_ALLOC;
    }
    if (rc == FA_OK)
        rc = launch_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, di, ws,
                             static_cast<char*>(ws) + z.zero_bytes(), st, 0, nullptr, 0, layout);
    const cudaError_t fe = cudaFreeAsync(ws, st);
    if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(workspace)", fe);
    return rc;
}

int fa_bwd_heads(const void* q, const void* k, const void* v, const void* o_bf16, const float* o_fp32,
                 const float* lse, const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 int causal, float scale, const int* head_modes, fa_stream_t stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dO) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv))
        return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, 0);
    if (rc) return rc;
    uint64_t mask[3];
    if ((rc = check_head_modes(head_modes, H, mask))) return rc;
    if (((mask[0] | mask[1]) && !aligned16(o_bf16)) || (mask[2] && !aligned16(o_fp32))) return FA_ERR_INVALID_ARG;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    const BwdSizes z = bwd_sizes(B * H, N, d);
    const size_t ws_bytes = z.zero_bytes() + z.row_bytes();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const char* fail = std::getenv("FA_TEST_FAIL_ALLOC");
    if (fail && fail[0] == '1') return FA_ERR_ALLOC;
    reserve_pool(di, ws_bytes);
    void* ws = nullptr;
    cudaError_t ae = cudaMallocAsync(&ws, ws_bytes, st);
    if (ae != cudaSuccess || !ws) {
        fa::set_error("cudaMallocAsync(workspace)", ae);
        cudaGetLastError();
        return FA_ERR_ALLOC;
    }
    // delta of each head from its own stored output: o_fp32 for the heads in
    // mode 2, o_bf16 for the others (a head's o is never read otherwise)
    const void* o_any = (mask[0] | mask[1]) ? o_bf16 : static_cast<const void*>(o_fp32);
    if (rc == FA_OK)
        rc = launch_backward(q, k, v, o_any, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, 0, di, ws,
                             static_cast<char*>(ws) + z.zero_bytes(), st, 0, o_fp32,
                             mask[2] ? mask[2] : 0);
    const cudaError_t fe = cudaFreeAsync(ws, st);
    if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(workspace)", fe);
    return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward with delta formed from O recomputed in FP32 (the forward in mode 2
// into a workspace), or from the caller's o.
int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
              void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, int mode,
              int delta_source, fa_stream_t stream) {
    if (delta_source == FA_DELTA_STORED_O)
        return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, stream);
    if (delta_source != FA_DELTA_RECOMPUTED_O_FP32 && delta_source != FA_DELTA_FROM_DP_P) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dO) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv))
        return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const char* fail = std::getenv("FA_TEST_FAIL_ALLOC");
    if (fail && fail[0] == '1') return FA_ERR_ALLOC;
    if (delta_source == FA_DELTA_FROM_DP_P) {
        // delta = rowsum(dP o P) from a pre-pass into the backward's row
        // workspace; the stored o is not read
        const int BH = B * H;
        const int Npad = (N + fa::kBlockM - 1) / fa::kBlockM * fa::kBlockM;
        const BwdSizes z = bwd_sizes(BH, N, d);
        reserve_pool(di, z.zero_bytes() + z.row_bytes());
        void* ws = nullptr;
        cudaError_t ae = cudaMallocAsync(&ws, z.zero_bytes() + z.row_bytes(), st);
        if (ae != cudaSuccess || !ws) {
            fa::set_error("cudaMallocAsync(workspace)", ae);
            cudaGetLastError();
            return FA_ERR_ALLOC;
        }
        float* rows = reinterpret_cast<float*>(static_cast<char*>(ws) + z.zero_bytes());
        if (rc == FA_OK) {
            fa::DeltaPdpArgs pa{};
            pa.q = q;
            pa.k = k;
            pa.v = v;
            pa.dout = dO;
            pa.lse = lse;
            pa.delta = rows + static_cast<size_t>(BH) * Npad;
            pa.BH = BH;
            pa.N = N;
            pa.Npad = Npad;
            pa.d = d;
            pa.causal = causal;
            pa.scale = scale;
            if (fa::launch_delta_pdp(pa, st) != cudaSuccess) rc = FA_ERR_CUDA;
        }
        // o is not read: delta is given; pass a valid pointer for the unused argument
        if (rc == FA_OK)
            rc = launch_backward(q, k, v, dO, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, 0, di, ws, rows, st, 1);
        const cudaError_t fe = cudaFreeAsync(ws, st);
        if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(workspace)", fe);
        return rc;
    }
    const size_t o_bytes = static_cast<size_t>(B) * H * N * d * sizeof(float);  // a multiple of 256
    const size_t lse_bytes = static_cast<size_t>(B) * H * N * sizeof(float);
    void* ws = nullptr;
    cudaError_t ae = cudaMallocAsync(&ws, o_bytes + lse_bytes, st);
    if (ae != cudaSuccess || !ws) {
        fa::set_error("cudaMallocAsync(recomputed O)", ae);
        cudaGetLastError();
        return FA_ERR_ALLOC;
    }
    float* o32 = static_cast<float*>(ws);
    // lse32 only receives the forward's LSE output, which the call requires.
    // The backward below takes the caller's lse on purpose: P is recomputed
    // from the same LSE as in the stored-O backward, so only delta's source
    // differs between the two.
    float* lse32 = reinterpret_cast<float*>(static_cast<char*>(ws) + o_bytes);
    rc = fa_fwd_ex(q, k, v, o32, lse32, B, H, N, d, causal, scale, FA_MODE_FP32_OUT, nullptr, stream);
    if (rc == FA_OK) rc = fa_bwd(q, k, v, o32, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, FA_MODE_FP32_OUT, stream);
    const cudaError_t fe = cudaFreeAsync(ws, st);
    if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(recomputed O)", fe);
    return rc;
}

// Allocation-free backward: the workspace is a file-scope device array.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];
// fixed split: the zero region first, the row region in the last 2 MiB
constexpr size_t kNoallocRowBytes = 2u * 1024u * 1024u;
constexpr size_t kNoallocZeroBytes = FA_NOALLOC_SCRATCH_BYTES - kNoallocRowBytes;

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device.  In host code
// g_noalloc_scratch names a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.  That
// lookup must not happen inside a stream capture, so a first call on a device
// made while `stream` is capturing is refused.
int noalloc_scratch(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) {
        fa::set_error_msg("fa_bwd_noalloc", "device index exceeds the library's device table (64)");
        return FA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            cudaGetLastError();
            fa::set_error_msg("fa_bwd_noalloc",
                              "the first call on a device looks up the scratch address and must precede stream capture");
            return FA_ERR_INVALID_ARG;
        }
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return cuda_fail("cudaGetSymbolAddress(scratch)", e);
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, int mode,
                   fa_stream_t stream) {
    if (!bwd_pointers_ok(q, k, v, o, lse, dO, dq, dk, dv)) return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    const BwdSizes z = bwd_sizes(B * H, N, d);
    if (z.zero_bytes() > kNoallocZeroBytes || z.row_bytes() > kNoallocRowBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "needs %zu + %zu bytes of scratch, the static limit is %zu + %zu bytes (FA_NOALLOC_SCRATCH_BYTES)",
                 z.zero_bytes(), z.row_bytes(), kNoallocZeroBytes, kNoallocRowBytes);
        fa::set_error_msg("fa_bwd_noalloc", msg);
        return FA_ERR_INVALID_ARG;
    }
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    void* ws = nullptr;
    if ((rc = noalloc_scratch(static_cast<cudaStream_t>(stream), &ws))) return rc;
    // The zero region (the dQ accumulator) is cleared by the first kernel of
    // every call; the row region sits at the end of the array.
    return launch_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, mode, di, ws,
                           static_cast<char*>(ws) + kNoallocZeroBytes, static_cast<cudaStream_t>(stream));
}

int fa_tie_stats(const void* q, const void* k, const void* v, const void* o, int B, int H, int N, int d,
                 int causal, float scale, int mode, int32_t* tie_count, float* pv_err, int32_t* p_one,
                 fa_stream_t stream) {
    return fa_tie_stats_ex(q, k, v, o, B, H, N, d, causal, scale, mode, nullptr, tie_count, pv_err, p_one,
                           nullptr, nullptr, stream);
}

int fa_tie_stats_ex(const void* q, const void* k, const void* v, const void* o, int B, int H, int N, int d,
                    int causal, float scale, int mode, const fa_stab_params_t* params, int32_t* tie_count,
                    float* pv_err, int32_t* p_one, const void* dO, float* delta_err, fa_stream_t stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(tie_count) ||
        !aligned16(pv_err) || (p_one && !aligned16(p_one)) || (delta_err && (!aligned16(delta_err) || !aligned16(dO))))
        return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    float beta = 0.f, eps = 0.f;
    if ((rc = check_params(params, &beta, &eps))) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    const int BH = B * H;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const fa::RowLayout lay = layout_of(FA_LAYOUT_BHND, H, N, d);
    CUtensorMap mq, mk, mv;
    if (make_rows_map(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64) ||
        make_rows_map(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lay, B, N, d, 64))
        return FA_ERR_CUDA;
    fa::FwdArgs a{};
    a.tm_q = &mq;
    a.tm_k = &mk;
    a.tm_v = &mv;
    a.tm_o = &mq;  // not read: the statistics variant writes no O
    a.o = nullptr;
    a.lse = nullptr;
    a.tie_count = tie_count;
    a.p_one = p_one;
    a.beta = beta;
    a.BH = BH;
    a.N = N;
    a.d = d;
    a.causal = causal;
    a.mode = mode;
    a.scale = scale;
    a.scale_log2 = log2e_times(scale);
    a.status = di->status;
    a.num_sms = di->num_sms;
    a.H = H;
    a.lay = lay;
    // A tolerance: the near-tie counts (and, in mode 1, each row's fixed
    // shift) from the row pre-pass (stream-ordered workspace, B*H*N*8 bytes).
    void* ws = nullptr;
    if (eps != 0.f) {
        const size_t nrow = static_cast<size_t>(BH) * N;
        cudaError_t ae = cudaMallocAsync(&ws, nrow * (sizeof(float) + sizeof(int32_t)), st);
        if (ae != cudaSuccess || !ws) {
            fa::set_error("cudaMallocAsync(row statistics)", ae);
            cudaGetLastError();
            return FA_ERR_ALLOC;
        }
        float* shift = static_cast<float*>(ws);
        int32_t* rs = reinterpret_cast<int32_t*>(shift + nrow);
        if (mode == FA_MODE_STABILISED) a.shift = shift;
        a.rs_in = rs;
        rc = launch_row_pass(q, k, BH, N, d, causal, scale, mode, beta, eps, shift, rs, st, lay);
    }
    if (rc == FA_OK && fa::launch_fwd(a, true, st) != cudaSuccess) rc = FA_ERR_CUDA;
    if (ws) {
        const cudaError_t fe = cudaFreeAsync(ws, st);
        if (fe != cudaSuccess && rc == FA_OK) rc = cuda_fail("cudaFreeAsync(row statistics)", fe);
    }
    if (rc != FA_OK) return rc;
    fa::StatsArgs s{};
    s.q = q;
    s.k = k;
    s.v = v;
    s.o = o;
    s.pv_err = pv_err;
    s.dout = dO;
    s.delta_err = delta_err;
    s.BH = BH;
    s.N = N;
    s.d = d;
    s.causal = causal;
    s.mode = mode;
    s.scale = scale;
    s.status = di->status;
    return fa::launch_pv_err(s, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_delta_error_split(const void* q, const void* k, const void* v, const void* o, const void* dO, int B, int H,
                         int N, int d, int causal, float scale, int mode, const fa_stab_params_t* params,
                         float* err_one, float* err_rest, float* err_out, fa_stream_t stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
        !aligned16(err_one) || !aligned16(err_rest) || !aligned16(err_out))
        return FA_ERR_INVALID_ARG;
    int rc = check_common(B, H, N, d, causal, scale, mode);
    if (rc) return rc;
    float beta = 0.f, eps = 0.f;
    if ((rc = check_params(params, &beta, &eps))) return rc;
    DeviceInfo* di = nullptr;
    if ((rc = device_info(&di))) return rc;
    fa::SplitArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dout = dO;
    a.err_one = err_one;
    a.err_rest = err_rest;
    a.err_out = err_out;
    a.BH = B * H;
    a.N = N;
    a.d = d;
    a.causal = causal;
    a.mode = mode;
    a.scale = scale;
    a.beta = beta;
    a.eps = eps;
    return fa::launch_delta_split(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_device_status(fa_stream_t stream, int reset) {
    DeviceInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (reset && h != 0) {
        const int zero = 0;
        if (cudaMemcpy(di->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (h & 1) return FA_ERR_TIMEOUT;
    return h == 0 ? FA_OK : FA_ERR_NONFINITE;
}

}  // extern "C"
