/*
 * dsa.h -- C ABI of the GB300 (sm_103a) sparse MLA ("DSA") attention library.
 *
 * The operation: token t, query head h.
 *   The valid slots of token t are the positions j < W with
 *     0 <= topk_idxs[t, j] < S_kv,
 *   and also j < topk_length[t] when a length array is given.
 *     - cuDNN frontend "DSA backward SM90: fix three top-k and
 *       attention-sink boundary failures", Why item 2.
 *     - cuDNN frontend "DSA bwd SM100 fix dropped dKV gradients when topk
 *       width > total_S_kv": a column position >= S_kv is not invalid.
 *   s_j = scale * q[t,h,:] . kv[idx_j,:]  over all D = d_qk columns.
 *   lse[t,h] = log sum_j exp(s_j)  (natural log; the sink is not included).
 *   out[t,h,:] = sum_j exp(s_j) / (sum_j exp(s_j) + exp(sink[h])) * kv[idx_j, 0:512]
 * Every head uses the same KV tensor, whose first 512 columns are V
 * (flash-attention "[CuTe, SM100] Support 1..128 Q heads in sparse MLA via
 * in-kernel TMA padding", Agent Notes).  Rows are D = d_qk = 576 columns
 * (512 V + 64 rope), or 512 with no rope part, the width that page's
 * section "Performance at DeepSeek-V4 shapes" measures.  The backward takes the loss
 * sum(dout * out) and returns dq, dkv (summed over every token and head
 * that gathered a row) and d_sink (cuDNN page above, "Not addressed" and
 * Testing).
 *
 * Conventions, for every entry point:
 *  - Tensors are dense and row-major.  Device pointers are 16-byte aligned,
 *    else DSA_ERR_ALIGNMENT.
 *  - The caller owns every buffer.  The library never allocates device
 *    memory.  Its only host state is set up on first use on each device:
 *    each kernel's shared-memory limit, and the device address of
 *    dsa_bwd_no_alloc's array.  Make a first call on a device before any
 *    stream capture there.  A cudaDeviceReset invalidates that state, and
 *    the library does not notice it: do not reset a device on which the
 *    library has been used while the library stays loaded.
 *  - All work is queued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and the calls return before it finishes.
 *  - Argument and shape errors are returned before anything is launched.
 *    A failed launch returns DSA_ERR_CUDA.
 *  - An index that fails the validity rule is data, not an error: it is
 *    masked.
 *  - An empty row (no valid slot, including topk_length <= 0) gives out = 0,
 *    lse = -FLT_MAX, dq = 0, and adds nothing to dkv.
 *  - topk_length > W is treated as W.
 *  - A NULL sink means no sink, i.e. sink = -inf.
 *  - T = 0 is a no-op.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,    /* null pointer, bad size or field */
  DSA_ERR_UNSUPPORTED = 2,    /* valid request this build does not handle */
  DSA_ERR_ALIGNMENT = 3,      /* a device pointer is not 16-byte aligned */
  DSA_ERR_WORKSPACE = 4,      /* workspace missing or too small */
  DSA_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
  DSA_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up waiting on a barrier */
  DSA_ERR_RANGE = 7           /* DSA_FLAG_DETERMINISTIC: a dkv row may have
                                 left the fixed-point accumulator's range */
} dsa_status_t;

typedef struct {
  int32_t T;       /* query tokens, >= 0                                   */
  int32_t H;       /* query heads, 1..128                                  */
  int32_t S_kv;    /* KV rows, >= 1, with d_qk * S_kv < 2^31               */
  int32_t W;       /* index slots per token, >= 1                         */
  int32_t d_qk;    /* q/kv row width D: 576 (512 V + 64 rope) or 512 (V)  */
  int32_t d_v;     /* V width (leading columns of kv); must be 512         */
  float scale;     /* softmax scale applied to q.kv (e.g. 1/sqrt(576))     */
  uint32_t flags;  /* OR of DSA_FLAG_DELTA_RESIDUAL, DSA_FLAG_DETERMINISTIC  */
} dsa_problem_t;

/*
 * DSA_FLAG_DELTA_RESIDUAL: a forward output that carries about fp32 O.
 * With this flag, `out` points to 2*T*H*512 bf16 values: the rounded
 * output [T, H, 512] followed by its rounding residual bf16(O - bf16(O))
 * [T, H, 512].
 *   - dsa_fwd writes both halves.
 *   - dsa_bwd takes its first delta estimate from their sum.
 * This is the forward-side fix that the cuDNN page "DSA backward SM90: fix
 * three top-k and attention-sink boundary failures" ("Not addressed") names
 * for the delta error of a bf16 out.  The backward no longer needs it: it
 * forms the exact delta itself (see dsa_bwd), so the flag only shrinks the
 * correction it applies.  The flag must be the same in the forward and the
 * backward call.
 */
#define DSA_FLAG_DELTA_RESIDUAL 1u

/*
 * DSA_FLAG_DETERMINISTIC: bitwise reproducible dkv (backward only).
 * By default the backward scatter-adds each token's dkv rows with fp32
 * atomics, so their order, and the last bits of dkv, change from run to
 * run.  The pages name both designs (an atomic one on SM90 and a separate
 * reduction on SM100).  With this flag the adds are 64-bit integer adds of
 * round(v * 2^32).  Integer addition is order-independent, so dkv is the
 * same bits every run; dq and d_sink are deterministic in both modes.
 *   - Resolution 2^-32 (2.3e-10) per add; every dkv element must stay
 *     below 2^31 in magnitude.
 *   - Range check: every element of KV row r receives n_r adds (the valid
 *     slots naming r), each at most m in magnitude (m: the largest |add|
 *     of the call), so its sum is bounded by n_r * m.  The backward counts
 *     n_r, tracks m, and where n_r * m reaches 2^31 the row may have
 *     wrapped: the call still completes, and the next dsa_device_status
 *     returns DSA_ERR_RANGE (dkv is then not to be trusted).  The bound is
 *     conservative: no row that passes it can have wrapped.
 *   - The dkv accumulator in the workspace takes 8 bytes per element
 *     instead of 4, plus 4 bytes per KV row for the range check
 *     (dsa_bwd_workspace_bytes accounts for both).
 * Ignored by dsa_fwd.
 */
#define DSA_FLAG_DETERMINISTIC 2u

/*
 * Forward.  Shapes and types (all device pointers):
 *   q            bf16  [T, H, D]     (D = d_qk: 576, or 512 with no rope part)
 *   kv           bf16  [S_kv, D]
 *   topk_idxs    int32 [T, W]
 *   topk_length  int32 [T], or NULL for the non-compact encoding
 *                (-1 marks unused slots)
 *   sink         fp32  [H], natural-log logits, or NULL
 *   out          bf16  [T, H, 512]  (written; [2, T, H, 512] with
 *                                    DSA_FLAG_DELTA_RESIDUAL)
 *   lse          fp32  [T, H]       (written)
 * One kernel launch.  Limits of this build: W <= 2048.
 */
dsa_status_t dsa_fwd(const dsa_problem_t* problem, const void* q, const void* kv,
                     const int32_t* topk_idxs, const int32_t* topk_length, const float* sink,
                     void* out, float* lse, void* stream);

/*
 * Bytes of device workspace that dsa_bwd needs for `problem`.  Returns 0 on
 * an invalid problem.  The workspace holds:
 *   - the dkv accumulator             [S_kv, D], fp32 (int64 with
 *                                     DSA_FLAG_DETERMINISTIC);
 *   - the compacted index lists       [T, W] and their counts [T];
 *   - per-(t,h) fp32 rows: lse*log2(e), sigma(lse - sink), delta, the
 *     d_sink terms and the delta correction;
 *   - the dS'/P scratch that the main stage writes and the finalize stage
 *     reads: bf16 [T, ceil(W / 128), 64 * ceil(H / 32), 128].
 */
size_t dsa_bwd_workspace_bytes(const dsa_problem_t* problem);

/*
 * Backward of the loss sum(dout * out).  Inputs are as for dsa_fwd, plus:
 *   out    bf16 [T, H, 512]  the forward output (with DSA_FLAG_DELTA_RESIDUAL
 *                            [2, T, H, 512] as written by dsa_fwd)
 *   lse    fp32 [T, H]       the forward's lse
 *   dout   bf16 [T, H, 512]
 * Outputs, all overwritten, never accumulated:
 *   dq     bf16 [T, H, D]
 *   dkv    bf16 [S_kv, D]    rows that no valid slot names are written as 0
 *   dsink  fp32 [H]          must be NULL exactly when sink is NULL
 * workspace: device memory of at least dsa_bwd_workspace_bytes(problem)
 * bytes, 256-byte aligned.  It is overwritten.
 * The call queues, in order: a memset, slot compaction, the dq kernel
 * (which also forms rowsum(dout * out) per row), the dkv kernel, the dkv
 * cast, and the d_sink reduce.
 * Delta.  The gradients use the exact delta[t,h] = sum_j P_j dP_j, the
 * accurate form in the cuDNN page's "Not addressed" table, not only
 * rowsum(dout * out) of the bf16 out (the FlashAttention identity), whose
 * rounding the one-hot rows of a saturated softmax turn into dq/dkv error.
 * No second pass over the top-k is needed: dS is formed with the delta of
 * out, and since the gradients are linear in delta, the difference is
 * applied to dq, dkv and d_sink once each token's sum of dS is known.
 */
dsa_status_t dsa_bwd(const dsa_problem_t* problem, const void* q, const void* kv,
                     const int32_t* topk_idxs, const int32_t* topk_length, const float* sink,
                     const void* out, const float* lse, const void* dout, void* dq, void* dkv,
                     float* dsink, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages that dsa_bwd queues, as separate calls for callers that
 * want to time or interleave them.  Each takes exactly dsa_bwd's arguments
 * and checks them the same way.  They must run in this order, on one stream
 * and with one workspace; together they equal one dsa_bwd call.
 *   dsa_bwd_preprocess  memset of the dkv accumulator and slot compaction
 *   dsa_bwd_main        rowsum(dout * out), P recompute, dS and dq for every
 *                       64-head group, which also stores the dS' and P tiles
 *                       into the workspace
 *   dsa_bwd_finalize    the dkv tile GEMM over all heads with its
 *                       scatter-add, the dkv fp32 -> bf16 cast and the
 *                       d_sink reduce
 */
dsa_status_t dsa_bwd_preprocess(const dsa_problem_t* problem, const void* q, const void* kv,
                                const int32_t* topk_idxs, const int32_t* topk_length,
                                const float* sink, const void* out, const float* lse,
                                const void* dout, void* dq, void* dkv, float* dsink,
                                void* workspace, size_t workspace_bytes, void* stream);
dsa_status_t dsa_bwd_main(const dsa_problem_t* problem, const void* q, const void* kv,
                          const int32_t* topk_idxs, const int32_t* topk_length,
                          const float* sink, const void* out, const float* lse, const void* dout,
                          void* dq, void* dkv, float* dsink, void* workspace,
                          size_t workspace_bytes, void* stream);
dsa_status_t dsa_bwd_finalize(const dsa_problem_t* problem, const void* q, const void* kv,
                              const int32_t* topk_idxs, const int32_t* topk_length,
                              const float* sink, const void* out, const float* lse,
                              const void* dout, void* dq, void* dkv, float* dsink,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_bwd without a workspace argument: the backward that allocates nothing.
 * There is no counterpart on the pages; this is a convenience of this
 * library.  It serves callers that cannot allocate device memory at call
 * time:
 *   - a plain C program that holds only its input and output buffers;
 *   - a serving loop under a fixed memory budget, where a cudaMalloc would
 *     synchronise the device.
 * Arguments, outputs and errors are those of dsa_bwd.  The workspace comes
 * from a fixed 64 MiB device array inside this library.  Every GPU that
 * loads the library holds that array until the process exits.
 *  - Size limit: if dsa_bwd_workspace_bytes(problem) exceeds 64 MiB, the
 *    call returns DSA_ERR_WORKSPACE and launches nothing.  64 MiB covers,
 *    for instance, T = 128 tokens at H = 128 with 640 slots per token.
 *  - Set-up: the first call on a device looks up the array's device address
 *    on the current device, once.  Make that first call before any stream
 *    capture.
 *  - Sharing: all calls share the one array, which keeps the last call's
 *    contents (the call clears what must start at zero).  Calls that overlap
 *    on the GPU, on different streams or from different threads, race on it.
 *    Serialise them.
 */
dsa_status_t dsa_bwd_no_alloc(const dsa_problem_t* problem, const void* q, const void* kv,
                              const int32_t* topk_idxs, const int32_t* topk_length,
                              const float* sink, const void* out, const float* lse,
                              const void* dout, void* dq, void* dkv, float* dsink, void* stream);

/*
 * Varlen batches.  B sequences share the call: their tokens are packed
 * along T and their KV rows along S_kv.
 *   cu_seqlens_q   int32 [B + 1], device: sequence b holds tokens
 *                  cu_seqlens_q[b] <= t < cu_seqlens_q[b + 1]
 *                  (cu_seqlens_q[0] = 0, cu_seqlens_q[B] = T)
 *   cu_seqlens_kv  int32 [B + 1], device: sequence b holds KV rows
 *                  cu_seqlens_kv[b] <= r < cu_seqlens_kv[b + 1]
 *                  (cu_seqlens_kv[0] = 0, cu_seqlens_kv[B] = S_kv)
 * The cuDNN frontend's DSA kernel is batched: it reads topk_length per
 * (batch, position) ("DSA backward SM90: fix three top-k and attention-sink
 * boundary failures", Why 1); the other pages run B = 1.  A token's indices count from the first KV row of its own
 * sequence: slot j is valid when 0 <= idx < (cu_seqlens_kv[b + 1] -
 * cu_seqlens_kv[b]) and j < topk_length[t], and then names KV row
 * cu_seqlens_kv[b] + idx.  The sink is per head, shared by all sequences;
 * dkv covers all S_kv rows.  The offsets are read on the device only: they
 * are expected to be non-decreasing; a token outside every sequence gets
 * no valid slot, and ranges are clamped into [0, S_kv], so malformed offsets
 * give wrong rows but never an access outside the tensors.
 */
typedef struct {
  int32_t B;                     /* sequences, >= 1 */
  const int32_t* cu_seqlens_q;   /* device, [B + 1], 4-byte aligned */
  const int32_t* cu_seqlens_kv;  /* device, [B + 1], 4-byte aligned */
} dsa_varlen_t;

/*
 * dsa_fwd and dsa_bwd for a varlen batch.  Arguments, layouts, outputs and
 * errors are theirs, with T and S_kv the packed totals; `varlen` must not be
 * NULL (DSA_ERR_INVALID_ARG).  The workspace of dsa_bwd_varlen is sized by
 * dsa_bwd_workspace_bytes(problem) as for one sequence of the packed sizes.
 */
dsa_status_t dsa_fwd_varlen(const dsa_problem_t* problem, const dsa_varlen_t* varlen,
                            const void* q, const void* kv, const int32_t* topk_idxs,
                            const int32_t* topk_length, const float* sink, void* out, float* lse,
                            void* stream);
dsa_status_t dsa_bwd_varlen(const dsa_problem_t* problem, const dsa_varlen_t* varlen,
                            const void* q, const void* kv, const int32_t* topk_idxs,
                            const int32_t* topk_length, const float* sink, const void* out,
                            const float* lse, const void* dout, void* dq, void* dkv, float* dsink,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Slot decode and compaction: the first step of both passes, exposed so
 * that callers can check it bit-exactly.  For each token, the valid KV rows
 * are written to idx_out[t, 0:count) in slot order and the count to
 * count_out[t].  idx_out[t, count:W) is left unspecified.
 *   idx_out    int32 [T, W]  (device)
 *   count_out  int32 [T]     (device)
 */
dsa_status_t dsa_topk_compact(const dsa_problem_t* problem, const int32_t* topk_idxs,
                              const int32_t* topk_length, int32_t* idx_out, int32_t* count_out,
                              void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * word.  Returns:
 *   DSA_ERR_DEVICE_TIMEOUT  a kernel gave up waiting on one of its own
 *                           barriers (outputs of that call are garbage);
 *   DSA_ERR_RANGE           a DSA_FLAG_DETERMINISTIC backward failed its
 *                           range check (its dkv is not to be trusted);
 *   DSA_ERR_CUDA            the stream reported an error;
 *   DSA_OK                  otherwise.
 */
dsa_status_t dsa_device_status(void* stream);

/*
 * Self-test of the bounded waits, for tests of a caller's failure handling;
 * it computes nothing.  Every wait inside this library's kernels gives up
 * after a time limit (2 s), records DSA_ERR_DEVICE_TIMEOUT in the library's
 * device error word and lets the kernel return, so that a lost arrival
 * never hangs the GPU.  This call queues one small kernel on `stream` with
 * two waits on barriers that nothing completes: one with a limit of
 * `limit_us` microseconds (1 .. 1000000, else DSA_ERR_INVALID_ARG), one
 * with the ordinary limit, which the first one's abort flag ends early.
 * The next dsa_device_status then returns DSA_ERR_DEVICE_TIMEOUT (and
 * clears the word); the context stays usable.
 */
dsa_status_t dsa_wait_selftest(uint32_t limit_us, void* stream);

/* Static English text for a status code. */
const char* dsa_status_string(dsa_status_t status);

/* ABI version of this library (major * 100 + minor). */
int dsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
