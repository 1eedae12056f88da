/*
 * fa.h -- C ABI of the GB300 (sm_103a) flash-attention library (libfa.so).
 *
 * The operation is the attention forward and backward studied in "Why
 * Low-Precision Transformer Training Fails: An Analysis on Flash Attention"
 * (arXiv 2510.04212), in three numerical modes:
 *
 *   FA_MODE_BASELINE    safe softmax, section 3.4.4: Pbar = exp(S - rowmax S),
 *                       Obar = Pbar V, O = Obar / rowsum(Pbar); O stored BF16.
 *   FA_MODE_STABILISED  the stabilised safe softmax of section 3.4.5: with
 *                       rm = rowmax(S) and rs = number of keys whose raw score
 *                       equals rm exactly, the shift is beta*rm if rm > 0 and
 *                       rs > 1, 0 if rm < 0 and rs > 1, rm otherwise (beta = 2,
 *                       the value of the paper's Figure 7 runs, unless
 *                       fa_fwd_ex / fa_tie_stats_ex set another); O stored BF16.
 *                       The result equals the baseline's in exact arithmetic.
 *   FA_MODE_FP32_OUT    as the baseline, but O is stored in FP32 (the
 *                       "compute O in FP32 in the forward" isolation
 *                       experiment of section 3.4.2, and the FP32 attention
 *                       output practice described on the practices page).
 *
 * Shapes and layouts (all tensors contiguous, row-major):
 *   q, k, v, dO, dq, dk, dv : BF16 [B, H, N, d]
 *   o                       : BF16 [B, H, N, d] in modes 0 and 1,
 *                             FP32 [B, H, N, d] in mode 2
 *   lse                     : FP32 [B, H, N], natural log of
 *                             sum_j exp(scale * q_i . k_j) over visible keys
 *   S = scale * Q K^T with scale > 0; with causal = 1, key j is visible to
 *   query i iff j <= i (queries and keys share the index range 0..N-1).
 *   Supported: d in {64, 128}; 1 <= N <= 8388480; B*H*N*d < 2^31.
 *
 * Ownership: the caller allocates every buffer on the current CUDA device and
 * keeps ownership; device pointers must be 16-byte aligned.  The library
 * keeps no reference to any argument after a call returns.
 *
 * Asynchrony: every call only enqueues work on `stream` (NULL = the legacy
 * default stream) and returns without synchronising.  Errors inside a kernel
 * surface at the caller's next synchronisation, as for any CUDA launch;
 * kernels also record bounded-wait timeouts in a device status word that
 * fa_device_status() reads.
 *
 * Errors: every entry point returns an fa_status_t.  Arguments are checked
 * before anything is enqueued; on a non-zero status nothing was launched.
 * No entry point throws, aborts or exits.
 */
#ifndef FA_H_
#define FA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
    FA_MODE_BASELINE = 0,
    FA_MODE_STABILISED = 1,
    FA_MODE_FP32_OUT = 2
} fa_mode_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, causal/mode/scale out of range */
    FA_ERR_UNSUPPORTED = 2, /* d not in {64,128}, or the current device is not sm_103 */
    FA_ERR_ALLOC = 3,       /* a workspace allocation failed */
    FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, tensor map) */
    FA_ERR_TIMEOUT = 5,     /* a kernel gave up on a bounded wait (fa_device_status) */
    FA_ERR_NONFINITE = 6    /* a forward produced a row whose LSE (so its output) is not
                               finite (fa_device_status) */
} fa_status_t;

/*
 * fa_fwd -- attention forward (section 3.4.4 equations; section 3.4.5 shift in
 * mode 1).  Reads q, k, v; writes o and lse.  Tiles: 128 queries x 128 keys;
 * the online (tiled) softmax keeps per row the running max M, the running
 * number C of keys equal to M, and the shift m = f(M, C) of the mode, and
 * rescales the accumulator whenever m changes, so the final shift is the one
 * the untiled rule gives.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, int causal, float scale, int mode,
           fa_stream_t stream);

/*
 * Parameters of the stabilised softmax (mode 1; section 3.4.5, "The modified
 * safe softmax"):
 *   beta : the shift factor of rows with a positive, repeated maximum
 *          (m = beta*rm).  The section requires beta > 1 and names [2, 8] as
 *          the range the authors use; beta = 2 is the value of its Figure 7
 *          runs.  Finite values > 1 are accepted.  A large beta on a row with
 *          a large positive repeated maximum underflows every Pbar of that row
 *          (exp(-(beta-1)*scale*rm) below the FP32 range), and O then is not
 *          finite; the section restricts the rule to rows where the plain
 *          softmax is stable.
 *   eps  : the tolerance of the tie test, in scaled units: rs counts the keys
 *          with scale*(rm - q.k) <= eps.  eps = 0 counts exact ties of the
 *          FP32 raw scores, tracked through the tiled forward with a running
 *          maximum and count.  eps > 0 (the section uses about 1e-3): a key
 *          counted within eps of a running maximum can drop out of range when
 *          a later key tile raises the maximum, so the whole row is needed
 *          first.  A pre-pass on CUDA cores (FP32 scores, one fixed summation
 *          order) finds each row's rm, rs and shift; the tensor-core forward
 *          then uses that shift from its first key tile on.  Costs a
 *          stream-ordered workspace of B*H*N*4 bytes (fa_fwd_ex) or B*H*N*8
 *          bytes (fa_tie_stats_ex), cudaMallocAsync on `stream` (FA_ERR_ALLOC
 *          if that fails), and two extra passes of QK^T on CUDA cores.
 * A NULL pointer selects the defaults (beta = FA_STAB_BETA_DEFAULT, eps = 0).
 * Modes 0 and 2 check the parameters but do not use them.
 */
typedef struct {
    float beta;
    float eps;
} fa_stab_params_t;
#define FA_STAB_BETA_DEFAULT 2.0f

/*
 * fa_fwd_ex -- fa_fwd with explicit stabilised-softmax parameters.
 * FA_ERR_INVALID_ARG if beta is not a finite value > 1 or eps is negative or
 * not finite.  Otherwise as fa_fwd (plus the eps > 0 pre-pass in mode 1).
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int N, int d, int causal, float scale, int mode,
              const fa_stab_params_t* params, fa_stream_t stream);

/*
 * fa_bwd -- attention backward from the saved LSE (P is recomputed as
 * exp(S - LSE)); delta = rowsum(dO o O) uses the stored o of the same mode
 * (BF16 in modes 0/1, FP32 in mode 2), dP = dO V^T, dS = scale * P o (dP -
 * delta), dQ = dS K (sections 3.4.2-3.4.3), dK = dS^T Q, dV = P^T dO.
 * Reads q, k, v, o, lse, dO; writes dq, dk, dv (BF16, FP32 accumulation).
 * When the previous kernel in `stream` is this library's forward, the first
 * backward kernel starts reading dO while that forward finishes (o and lse
 * only after it has): dO must not overlap the forward's outputs.
 * Allocates a stream-ordered workspace (cudaMallocAsync on `stream`, freed on
 * `stream` before return; FA_ERR_ALLOC if that fails) of Z + R bytes, where
 * Z = B*H*N*d*4 (the FP32 dQ accumulator, cleared by the first kernel)
 * and R = 2*B*H*ceil(N/128)*128*4 (per-row LSE and delta terms).  The first
 * time a workspace size is seen on a device, the release threshold of the
 * device's current memory pool is raised to at least that size (never
 * lowered), so steady-state calls reuse pool memory instead of returning it
 * to the OS at every synchronisation.  Three kernels run in order on
 * `stream`: the per-row terms, the persistent main kernel (at most one CTA
 * per SM; every wait bounded, FA_ERR_TIMEOUT through fa_device_status if one
 * runs out), and the conversion of dQ to BF16.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dO, void* dq, void* dk, void* dv,
           int B, int H, int N, int d, int causal, float scale, int mode,
           fa_stream_t stream);

/*
 * fa_bwd_ex -- fa_bwd with a choice of the output that delta =
 * rowsum(dO o O) is formed from (section 3.4.2, "Isolation Experiments:
 * Narrowing Down the Failure Source"):
 *   FA_DELTA_STORED_O          the caller's o, as fa_bwd does (o in `mode`'s
 *                              dtype);
 *   FA_DELTA_RECOMPUTED_O_FP32 O recomputed inside the backward as P V in FP32:
 *                              the forward runs in FA_MODE_FP32_OUT into a
 *                              stream-ordered workspace of B*H*N*(d+1)*4 bytes
 *                              (cudaMallocAsync on `stream`, on top of
 *                              fa_bwd's), and delta is formed from it; o is
 *                              not read and may be NULL.
 *   FA_DELTA_FROM_DP_P         delta = rowsum(dP o P) (section 3.4.2, "Failure
 *                              is linked to the computation of delta"; the
 *                              delta substitution of section 5): equal to
 *                              rowsum(dO o O) in exact arithmetic, formed
 *                              without any output.  A pre-pass on CUDA cores
 *                              recomputes P = exp(scale*q.k - lse) and
 *                              dP = dO.v in FP32 over each row (compensated
 *                              sum) into fa_bwd's workspace; o is not read
 *                              and may be NULL, `mode` is only checked.
 * P is recomputed from the caller's lse in every case, so only delta's source
 * changes.  Other arguments and errors as fa_bwd; FA_ERR_INVALID_ARG for an
 * unknown delta_source.
 */
typedef enum {
    FA_DELTA_STORED_O = 0,
    FA_DELTA_RECOMPUTED_O_FP32 = 1,
    FA_DELTA_FROM_DP_P = 2
} fa_delta_source_t;
int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dO, void* dq, void* dk, void* dv,
              int B, int H, int N, int d, int causal, float scale, int mode,
              int delta_source, fa_stream_t stream);

/*
 * Layouts of the [*, N, d] tensors (q, k, v, o, dO, dq, dk, dv; lse stays
 * [B, H, N]):
 *   FA_LAYOUT_BHND  [B, H, N, d] contiguous (what every other entry point takes)
 *   FA_LAYOUT_BNHD  [B, N, H, d] contiguous (heads interleaved per position, as
 *                   a projection's output is laid out before any transpose)
 * fa_fwd_layout / fa_bwd_layout -- fa_fwd_ex / fa_bwd with a layout; the
 * kernels address the tensors in place (4-D tensor maps; no copy).
 * FA_ERR_INVALID_ARG for an unknown layout.  Otherwise as fa_fwd_ex / fa_bwd.
 */
enum { FA_LAYOUT_BHND = 0, FA_LAYOUT_BNHD = 1 };
int fa_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int N, int d, int causal, float scale, int mode,
                  const fa_stab_params_t* params, int layout, fa_stream_t stream);
int fa_bwd_layout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv,
                  int B, int H, int N, int d, int causal, float scale, int mode,
                  int layout, fa_stream_t stream);

/*
 * Per-head modes (section 5, "Head-wise high-precision substitution": the
 * FP32 output only for the heads implicated in the failure).
 *
 * fa_fwd_heads -- the forward with a mode per head: head_modes is a host
 * array of H entries in {FA_MODE_BASELINE, FA_MODE_STABILISED,
 * FA_MODE_FP32_OUT}, the same for every batch; H <= 64 (FA_ERR_UNSUPPORTED
 * above).  The heads in modes 0 and 1 write BF16 O into o_bf16, those in mode
 * 2 FP32 O into o_fp32; both buffers are full [B,H,N,d] tensors of which only
 * their heads' slices are written (either may be NULL if no head uses it).
 * lse is written for every head.  params as fa_fwd_ex (used by mode-1 heads).
 * One forward launch per mode present, each over its own heads.
 *
 * fa_bwd_heads -- the matching backward: delta = rowsum(dO o O) of each head
 * from its own stored output (o_fp32 for mode-2 heads, o_bf16 otherwise);
 * everything else as fa_bwd (same workspace, one launch).
 *
 * Errors as fa_fwd / fa_bwd; FA_ERR_INVALID_ARG for a NULL head_modes or an
 * entry out of range.
 */
int fa_fwd_heads(const void* q, const void* k, const void* v, void* o_bf16, float* o_fp32,
                 float* lse, int B, int H, int N, int d, int causal, float scale,
                 const int* head_modes, const fa_stab_params_t* params, fa_stream_t stream);
int fa_bwd_heads(const void* q, const void* k, const void* v, const void* o_bf16,
                 const float* o_fp32, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                 float scale, const int* head_modes, fa_stream_t stream);

/*
 * fa_bwd_noalloc -- the same backward as fa_bwd, for callers that must not
 * allocate device memory: code that runs after a framework's caching
 * allocator has reserved (nearly) all of the GPU's memory, so a driver
 * allocation would fail or fragment it; latency-critical loops where an
 * allocation call may block or synchronise; deployments that forbid
 * allocation after start-up; and devices or setups without stream-ordered
 * memory pools.  (The paper has no counterpart; this is a deployment variant
 * of fa_bwd.)
 *
 * Instead of a cudaMallocAsync workspace it uses a fixed scratch array
 * compiled into this library, FA_NOALLOC_SCRATCH_BYTES (32 MiB) per device;
 * every GPU that loads the library holds that array until the process exits.
 * The caller still passes all inputs and outputs.  The array is split into a
 * 30 MiB part that holds fa_bwd's Z bytes (see fa_bwd) and a 2 MiB part that
 * holds its R bytes; problems whose Z or R does not fit (at d = 64, B*H*N
 * above about 122,000 rows) are rejected with FA_ERR_INVALID_ARG before
 * anything is enqueued (fa_last_error says why).  As in fa_bwd, the first
 * kernel clears the accumulator.  The first call on a device also looks up the
 * array's device address on that device; make that first call before any
 * stream capture (a first call made while `stream` is capturing is refused
 * with FA_ERR_INVALID_ARG).  All calls share the one array, so calls whose
 * execution overlaps on the GPU -- e.g. on two streams without an ordering
 * between them -- race on the scratch and give wrong results: serialise
 * them.  Allocates nothing and calls no allocating routine.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, int causal, float scale, int mode,
                   fa_stream_t stream);

/*
 * fa_tie_stats -- per-row diagnostics of the forward of `mode`:
 *   tie_count[r] : number of visible keys whose FP32 raw score q.k equals the
 *                  row maximum exactly (the rs of section 3.4.5 with eps = 0);
 *   pv_err[r]    : sum over the d columns of (o[r,c] - O_ref[r,c]), the signed
 *                  rounding error of the stored output, where O_ref is a
 *                  CUDA-core FP32 recomputation of softmax(S) V (two passes,
 *                  exact row max, compensated sums); o is the output of
 *                  fa_fwd for the same mode (section 3.4.4, "Isolating the
 *                  error to PV");
 *   p_one        : nullable; p_one[r] = number of BF16 Pbar entries equal to
 *                  1.0 fed to the PV product, p_one[B*H*N + r] = number of
 *                  keys whose final weight (Pbar times later rescale factors)
 *                  is exactly 1.0 (the condition of section 3.4.4, "Why
 *                  P[T,t] = 1 is the critical condition").
 * All three are [B, H, N] (p_one [2, B, H, N]); rows are r = (b*H + h)*N + i.
 */
int fa_tie_stats(const void* q, const void* k, const void* v, const void* o,
                 int B, int H, int N, int d, int causal, float scale, int mode,
                 int32_t* tie_count, float* pv_err, int32_t* p_one,
                 fa_stream_t stream);

/*
 * fa_tie_stats_ex -- fa_tie_stats with explicit stabilised-softmax parameters
 * (checked as by fa_fwd_ex), and optionally the error that the stored output
 * brings into the backward's delta = rowsum(dO o O):
 *   delta_err : nullable FP32 [B, H, N]; delta_err[r] = sum_c dO[r,c] *
 *               (o[r,c] - O_ref[r,c]) with the same FP32 reference O_ref as
 *               pv_err, i.e. delta_lp - delta_hp of section 3.4.4 ("Cause 2:
 *               Biased Rounding Error Leads to Positive (delta_lp -
 *               delta_hp)[T]"), O_ref standing in for the FP32 output O_hp;
 *   dO        : BF16 [B, H, N, d], read only when delta_err is set (then
 *               both must be 16-byte aligned device pointers).
 * The p_one counts of mode 1 follow beta and eps; o must come from fa_fwd_ex
 * with the same parameters.  With eps > 0, tie_count[r] is the row's
 * near-tie count rs (every mode), from the row pre-pass.
 */
int fa_tie_stats_ex(const void* q, const void* k, const void* v, const void* o,
                    int B, int H, int N, int d, int causal, float scale, int mode,
                    const fa_stab_params_t* params,
                    int32_t* tie_count, float* pv_err, int32_t* p_one,
                    const void* dO, float* delta_err,
                    fa_stream_t stream);

/*
 * fa_delta_error_split -- the decomposition of delta_lp - delta_hp for a
 * stored output o of `mode` (section 3.4.4, "Cause 2: Biased Rounding Error
 * Leads to Positive (delta_lp - delta_hp)[T]"; the quantitative decomposition
 * the page lists among the missing experiments).  Per row r, with the row's
 * shift m (the untiled rule of the mode with the parameters' beta and eps),
 * P_j = exp(scale*q.k_j - m), b_j = bf16(P_j), l = sum_j P_j and the FP32
 * reference probabilities p_j (exact row maximum, compensated sums):
 *   err_one[r]  = sum_c dO[r,c] sum_{j: b_j = 1}  (b_j / l - p_j) v_j[c]
 *   err_rest[r] = sum_c dO[r,c] sum_{j: b_j != 1} (b_j / l - p_j) v_j[c]
 *   err_out[r]  = sum_c dO[r,c] (o[r,c] - sum_j b_j v_j[c] / l)
 * so that err_one + err_rest + err_out = sum_c dO (o - O_ref), the delta_err
 * of fa_tie_stats_ex.  The split follows the untiled softmax (a key's
 * probability with the row's final shift); in the tiled forward a running
 * maximum may have been fed as 1 and rescaled later.  q, k, v, dO BF16
 * [B,H,N,d]; o BF16 (FP32 in mode 2); outputs FP32 [B,H,N].  Diagnostic: CUDA
 * cores, FP32, about (d/8 + 3) passes over each row's keys.
 */
int fa_delta_error_split(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, int B, int H, int N, int d, int causal,
                         float scale, int mode, const fa_stab_params_t* params,
                         float* err_one, float* err_rest, float* err_out,
                         fa_stream_t stream);

/*
 * fa_device_status -- synchronises `stream`, then returns FA_ERR_TIMEOUT if any
 * kernel of this library on the current device recorded a bounded-wait
 * timeout since the last reset, else FA_ERR_NONFINITE if a forward wrote a
 * row whose LSE is not finite (every Pbar of the row underflowed, e.g. a large
 * beta on a large repeated maximum; its O is then not finite either),
 * FA_ERR_CUDA if the synchronisation failed, else FA_OK.  reset != 0 clears
 * the recorded status.
 */
int fa_device_status(fa_stream_t stream, int reset);

/*
 * Per-kernel timing (instrumentation for benchmarks).  Between
 * fa_profile_start() and fa_profile_stop(), every kernel this library
 * launches on the calling thread's current device is bracketed by a pair of
 * CUDA events recorded on the launch stream.  fa_profile_stop() synchronises
 * those events and, for each kernel kind k < n (see FA_KERNEL_*), writes the
 * number of launches to launches[k] and their summed duration in
 * milliseconds to total_ms[k] (either may be NULL).  Events are created
 * lazily and reused; at most FA_PROFILE_MAX_LAUNCHES launches are recorded per
 * session (later ones are counted in launches[] but not timed, and
 * fa_profile_stop returns FA_ERR_ALLOC).  Not thread-safe across concurrent
 * callers.  Launches captured into a CUDA graph during a session record their
 * events as external event-record nodes (cudaEventRecordExternal): launch the
 * instantiated graph once, then stop the session, and the totals are that
 * launch's.
 */
enum {
    FA_KERNEL_FWD = 0,       /* forward (modes 0-2) */
    FA_KERNEL_FWD_STATS = 1, /* forward replay writing tie counts */
    FA_KERNEL_BWD_PRE = 2,   /* backward, first kernel: delta and LSE*log2(e) per row */
    FA_KERNEL_BWD_MAIN = 3,  /* backward, main kernel: the five-MMA loop */
    FA_KERNEL_DQ_CONVERT = 4,/* backward, last kernel: FP32 dQ accumulator -> BF16 */
    FA_KERNEL_PV_ERR = 5,    /* CUDA-core reference for pv_err */
    FA_KERNEL_COUNT = 6,
    FA_PROFILE_MAX_LAUNCHES = 65536
};
int fa_profile_start(void);
int fa_profile_stop(int n, int64_t* launches, double* total_ms);

/*
 * Description of the most recent CUDA failure behind an FA_ERR_CUDA (or
 * FA_ERR_ALLOC) returned on the calling thread: the failing step and the CUDA
 * error string, e.g. "bwd_main launch: too many resources requested for
 * launch".  Empty if none.  Thread-local static storage, valid until the next
 * call on this thread.
 */
const char* fa_last_error(void);

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
