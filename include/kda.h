/*
 * kda.h -- C ABI of libkda, Kimi Delta Attention (KDA) on NVIDIA GB300 (sm_103a).
 *
 * The operations are those of the Kimi K3 technical report:
 *   - bounded gate, section 2.1.1 Eq. 5 (the bias b of Eq. 2 sits inside the
 *     logit, as in the flash-linear-attention `lower_bound` gate quoted by the
 *     xuquant.com review of the report):
 *         g = g_min * Sigmoid(exp(A_log[h]) * (z + b[h])),   alpha = exp(g)
 *   - recurrence, section 2.1.1 Eq. 1 (decay before the delta update):
 *         S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *         o_t = scale * S_t^T q_t              (scale = 1 in the report)
 *   - chunkwise evaluation, section 2.1.1 Eq. 3 and Eq. 4 (parallel inside a
 *     chunk, recurrent across chunks), and the single-token decode step of
 *     section 5.4.2.
 *
 * Conventions shared by every entry point
 *   - Memory: every tensor pointer is a DEVICE pointer on the current CUDA
 *     device, owned by the caller.  The library allocates no device memory and
 *     frees nothing; the prefill scratch ("workspace") is passed in by the caller
 *     and sized by kda_chunk_fwd_workspace_size().  Tensors are dense,
 *     row-major ("C-contiguous") with the shapes stated below, and 16-byte
 *     aligned.
 *   - Layout: token-major [T, H, d] for per-token vectors (T = all tokens of all
 *     sequences packed back to back), [T, H] for beta, [H, d_k] for dt_bias,
 *     [H] for A_log, and [N, H, d_k, d_v] for recurrent states (row = key
 *     channel, column = value channel; each head's 128 x 128 state is one
 *     contiguous block, as in the paged state layout of section 5.4.1).
 *   - Types: kda_dtype_t selects the I/O type of q, k, v, z, beta and o (fp32 or
 *     bf16).  dt_bias, A_log and states are always fp32.  Arithmetic is fp32.
 *   - Streams: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns before it finishes.
 *   - Errors: every call validates its arguments on the host first and returns
 *     a kda_status_t; on failure it launches nothing.  Nothing aborts, traps or
 *     throws across this boundary.  Problems only visible on the device
 *     (inconsistent cu_seqlens contents, an out-of-range state index) set a
 *     device error word that kda_get_device_error() reads back and clears; the
 *     affected work items are skipped.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

#define KDA_ABI_VERSION 5

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,       /* NULL where a tensor is required, negative size, bad g_min */
    KDA_ERR_UNSUPPORTED_SHAPE = 2, /* head size or chunk size not built into this library */
    KDA_ERR_UNSUPPORTED_DTYPE = 3,
    KDA_ERR_MISALIGNED = 4,        /* a tensor pointer is not 16-byte aligned */
    KDA_ERR_WORKSPACE = 5,         /* workspace NULL or smaller than required */
    KDA_ERR_CUDA = 6,              /* a CUDA runtime call or launch failed */
    KDA_ERR_BAD_SEQLENS = 7,       /* (device) cu_seqlens not 0 = c_0 <= c_1 <= ... <= c_N = T */
    KDA_ERR_BAD_STATE_INDEX = 8,   /* (device) state_indices entry outside [0, num_slots) */
    KDA_ERR_NO_DEVICE = 9,         /* no current CUDA device of compute capability 10.3 */
    KDA_ERR_DEVICE_TIMEOUT = 10,   /* (device) a bounded wait inside a kernel gave up */
    KDA_ERR_BAD_TOKEN_COUNT = 11,  /* (device) n_replay / n_commit entry outside its range */
    KDA_ERR_NUMERIC = 12           /* (device, debug checks only) an output holds a NaN or an infinity */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Gate of the log-decay g (section 2.1.1).  Every entry point that takes z takes a gate_kind.
 *   KDA_GATE_LOWER_BOUND (0): Eq. 5, g = g_min * Sigmoid(exp(A_log[h]) * (z + b[h])) in (g_min, 0).
 *     The bound keeps every in-chunk decay factor inside bf16 range, which is what lets the
 *     bf16 d = 128 prefill run as dense tensor-core products.
 *   KDA_GATE_SOFTPLUS (1): the unbounded gate of the earlier design that Eq. 5 replaces,
 *     g = -exp(A_log[h]) * Softplus(z + b[h]) in (-inf, 0); g_min is ignored.  The prefill then
 *     runs on the fp32 CUDA-core path, which forms each in-chunk decay as exp(G_r - G_i) <= 1
 *     from the cumulative log-decays (never as a product of Gamma and 1 / Gamma), so no value
 *     of the gate overflows; a decay that underflows erases the state, as it should. */
typedef enum { KDA_GATE_LOWER_BOUND = 0, KDA_GATE_SOFTPLUS = 1 } kda_gate_kind_t;

/* ------------------------------------------------------------------ kda_gate
 * Eq. 5 (section 2.1.1): per-channel log-decay g = g_min * Sigmoid(exp(A_log[h]) * (z + b[h]))
 * (or the softplus gate, see kda_gate_kind_t) for every token, optionally followed by the chunk-local cumulative sum of
 * Eq. 3 in log space, G_r = sum_{i <= r} g_i, restarting at every chunk start
 * (chunks of `chunk_size` tokens aligned to each sequence's first token).
 */
typedef struct {
    int64_t T;                 /* tokens (all sequences packed) */
    int64_t N;                 /* sequences (>= 1 when T > 0; ignored when chunk_size == 0) */
    int32_t H;                 /* heads */
    int32_t dk;                /* key channels (any value >= 1) */
    kda_dtype_t dtype;         /* dtype of z */
    const void *z;             /* [T, H, dk] decay logit without bias */
    const float *dt_bias;      /* [H, dk] per-head bias b, or NULL for zero */
    const float *A_log;        /* [H] per-head log-scale A, or NULL for zero */
    float g_min;               /* lower bound of the log-decay, < 0 (the report uses -5); unused by
                                  KDA_GATE_SOFTPLUS */
    int32_t chunk_size;        /* 0: write g; > 0: write the chunk-local cumulative sum */
    const int32_t *cu_seqlens; /* [N + 1] sequence starts, or NULL for N equal lengths T / N */
    float *out;                /* [T, H, dk] fp32 output */
    int32_t gate_kind;         /* kda_gate_kind_t (0: Eq. 5) */
} kda_gate_args;

kda_status_t kda_gate(const kda_gate_args *args, struct CUstream_st *stream);

/* ------------------------------------------------------------- kda_chunk_fwd
 * Prefill: Eq. 1 over whole sequences, evaluated chunkwise as in Eq. 3 and
 * Eq. 4 (section 2.1.1).  Inside each chunk of C = 64 tokens the UT transform
 * yields U and W (pseudo-values V~ = U - W S), and outputs are
 * O = (Gamma * Q) S + Tril[(Q * Gamma)(K / Gamma)^T] V~; across chunks the
 * state is carried as S <- Diag(gamma^C) S + (K * gamma^C / Gamma)^T V~.
 * The gate of Eq. 5 is fused.  Chunks start at each sequence's first token;
 * the last chunk of a sequence may be shorter.
 *
 * Supported: d_k = d_v in {64, 128}; chunk_size 64 (0 selects 64).
 * bf16 with d_k = d_v = 128 runs on the tensor cores (tcgen05) with the bounded
 * gate and g_min >= -5.5; every other case runs on the fp32 CUDA-core path.
 * Empty sequences are allowed: their final state is their initial state (zero
 * without one), copied exactly.  An empty batch (T = 0) does only that and
 * reads no token pointer.
 */
typedef struct {
    int64_t T;                     /* tokens (all sequences packed) */
    int64_t N;                     /* sequences, >= 1 */
    int32_t H, dk, dv;             /* heads, key channels, value channels */
    kda_dtype_t dtype;             /* dtype of q, k, v, z, beta and o */
    const void *q, *k, *z;         /* [T, H, dk] (q and k as given: the kernels do not normalise) */
    const void *v;                 /* [T, H, dv] */
    const void *beta;              /* [T, H] write strength in (0, 1), used as given */
    const float *dt_bias;          /* [H, dk] or NULL (zero) */
    const float *A_log;            /* [H] or NULL (zero) */
    float g_min;                   /* < 0; the report uses -5 (unused by KDA_GATE_SOFTPLUS) */
    float scale;                   /* output scale; Eq. 1 has none (pass 1) */
    const int32_t *cu_seqlens;     /* [N + 1] device, or NULL for N sequences of T / N tokens */
    const int32_t *cu_seqlens_host;/* optional HOST copy of cu_seqlens (enables long-sequence
                                      splitting across SMs); NULL = plan from T, N alone */
    const float *initial_state;    /* [N, H, dk, dv] or NULL (zero state) */
    float *final_state;            /* [N, H, dk, dv] or NULL; may alias initial_state */
    void *o;                       /* [T, H, dv] output; must not alias an input */
    int32_t chunk_size;            /* 64, or 0 for the default (64) */
    /* Optional output epilogue (Eq. 6 without its projections; see kda_output_gate): when out_gate
     * is set, o receives Sigmoid(out_gate) * RMSNorm(o~) instead of the recurrent output o~ (the norm
     * taken on o~ rounded to the dtype of o, as kda_output_gate would read it).  The tensor-core path
     * applies it in its output pass before o is stored when the chains run as separate kernels; the
     * one-launch schedule (whose chains bound the call) and the fp32 path run a kda_output_gate pass
     * over o in place after the recurrence. */
    const void *out_gate;          /* [T, H, dv], dtype of o, 16-byte aligned, or NULL (no epilogue) */
    const float *out_norm_weight;  /* [H, dv] RMSNorm weight, 16-byte aligned, or NULL (ones) */
    float out_norm_eps;            /* RMSNorm epsilon, > 0 when out_gate is set */
    int32_t gate_kind;             /* kda_gate_kind_t (0: Eq. 5; KDA_GATE_SOFTPLUS runs the fp32 path) */
} kda_chunk_args;

/* Bytes of device scratch kda_chunk_fwd needs for these sizes (0 on invalid sizes).
 * Depends only on (T, N, H, dk, dv, dtype, chunk_size) and the presence of
 * cu_seqlens_host (pass has_host_seqlens = 1 when it will be given). */
size_t kda_chunk_fwd_workspace_size(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                    kda_dtype_t dtype, int32_t chunk_size,
                                    const int32_t *cu_seqlens_host);
/* The same for a given gate kind (kda_chunk_fwd_workspace_size is gate_kind 0; the softplus gate
 * takes the fp32 path, whose records are larger for bf16 d = 128).  The bf16 d = 128 tensor-core
 * prefill scales rows and keys by e^{G_r - G_p} against references at most 16 tokens away, exact while
 * 16 |g_min| stays inside fp32 range: with the bounded gate and g_min < -5.5 kda_chunk_fwd runs the
 * fp32 path instead, whose workspace is this function's value for KDA_GATE_SOFTPLUS. */
size_t kda_chunk_fwd_workspace_size_gate(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                         kda_dtype_t dtype, int32_t chunk_size,
                                         const int32_t *cu_seqlens_host, int32_t gate_kind);

/* workspace: device memory of at least kda_chunk_fwd_workspace_size() bytes,
 * 256-byte aligned, owned by the caller; its contents need no initialisation
 * and are garbage afterwards.  Calls that share a workspace must not overlap.
 * Stream capture: the one-launch and chain-team schedules publish their
 * per-chunk work through flags, and the producers take their items from a
 * counter, both tagged with a per-call number kept on the host, which a captured
 * graph would freeze; a call made while `stream` is being captured therefore
 * runs the flag-free separate kernels with a fixed split of the items (same
 * results, more launches), and its graph may be replayed with new contents in
 * the same buffers. */
kda_status_t kda_chunk_fwd(const kda_chunk_args *args, void *workspace, size_t workspace_bytes,
                           struct CUstream_st *stream);

/* ------------------------------------------------------ kda_recurrent_replay
 * Speculative decoding with replay (section 5.4, KDA decode kernel): instead of
 * keeping a state snapshot per draft position, only the draft tokens' projected
 * inputs are cached; the state of the accepted drafts is rebuilt on chip from
 * them, and the replayed tokens, the bonus token and the next draft window run
 * in one loop.  Per (sequence n, head h), starting from the committed state
 * S = state[slot(n), h]:
 *   1. replay tokens 0 .. n_replay[n] - 1 of the cached window (Eq. 1; no outputs);
 *   2. run the M new tokens in order (Eq. 1), writing o for each;
 *   3. write back the state reached after the replayed tokens and the first
 *      n_commit[n] new tokens (typically the bonus token); later new tokens are
 *      drafts: their outputs are written, their state is not.  When
 *      n_replay[n] + n_commit[n] = 0 the state is left untouched.
 * The state crosses HBM once (read) plus once (write) per call, whatever the
 * number of tokens.  Counts outside [0, R] / [0, M] set KDA_ERR_BAD_TOKEN_COUNT
 * on the device and skip that sequence.  Shapes as kda_recurrent_step.
 */
typedef struct {
    int64_t N;                     /* sequences */
    int32_t H, dk, dv;             /* heads; dk = dv in {64, 128} */
    kda_dtype_t dtype;             /* dtype of every token input and of o */
    int32_t R;                     /* cached tokens per sequence (replay window), >= 0 */
    const void *rq, *rk, *rz;      /* [N, R, H, dk] cached inputs (may be NULL when R == 0) */
    const void *rv;                /* [N, R, H, dv] */
    const void *rbeta;             /* [N, R, H] */
    const int32_t *n_replay;       /* [N] device: accepted cached tokens to replay, 0 .. R */
    int32_t M;                     /* new tokens per sequence (bonus token, then drafts), >= 1 */
    const void *q, *k, *z;         /* [N, M, H, dk] */
    const void *v;                 /* [N, M, H, dv] */
    const void *beta;              /* [N, M, H] */
    const int32_t *n_commit;       /* [N] device: new tokens whose state is committed, 0 .. M */
    const float *dt_bias;          /* [H, dk] or NULL */
    const float *A_log;            /* [H] or NULL */
    float g_min, scale;            /* as kda_recurrent_step */
    float *state;                  /* [num_slots, H, dk, dv] committed states, updated in place */
    const int32_t *state_indices;  /* [N] slot of each sequence, or NULL (slot n); distinct slots */
    int64_t num_slots;             /* 0 = N */
    void *o;                       /* [N, M, H, dv] outputs of the new tokens */
    int32_t gate_kind;             /* kda_gate_kind_t (0: Eq. 5) */
} kda_replay_args;

kda_status_t kda_recurrent_replay(const kda_replay_args *args, struct CUstream_st *stream);

/* ------------------------------------------------------------- kda_chunk_bwd
 * Backward pass of kda_chunk_fwd, for training (the FlashKDA kernels of section 5.1.1 serve
 * training; the report gives the forward only).  The gradients are the exact derivatives of the
 * chunkwise form of Eq. 3 and Eq. 4 (which equals Eq. 1): given dL/do and optionally dL/dS_T, it
 * returns dL/d of q, k, v, z, beta, dt_bias, A_log and the initial state.  Across chunks the
 * state's adjoint runs backwards, Lambda_in = Diag(gamma^C) Lambda + scale Q^^T dO - W^T dV~ with
 * dV~ = K~ Lambda + scale A^T dO; every other gradient is local to its chunk (the state entering
 * it, the Lambda leaving it and dO).  The forward quantities are recomputed (nothing is kept from
 * kda_chunk_fwd): the chunk-local quantities in fp32 on CUDA cores; with bf16 I/O at d_k = d_v = 128
 * the two chains and the value-channel contractions are tcgen05 products of bf16 operand images with
 * fp32 accumulation (fp32 I/O stays in fp32 throughout).  The gate's derivative (either gate kind)
 * is applied per token; dt_bias and A_log gradients are summed over all tokens
 * (and written, as zeros, when there are none: T = 0).  For an empty sequence the
 * initial state's gradient is its final state's (zero without one).
 * Supported: as kda_chunk_fwd (d_k = d_v in {64, 128}, chunk_size 64).
 */
typedef struct {
    int64_t T, N;                   /* tokens, sequences (as kda_chunk_fwd) */
    int32_t H, dk, dv;
    kda_dtype_t dtype;              /* dtype of every [T, ...] tensor below, inputs and gradients */
    const void *q, *k, *z;          /* [T, H, dk] forward inputs */
    const void *v;                  /* [T, H, dv] */
    const void *beta;               /* [T, H] */
    const float *dt_bias;           /* [H, dk] or NULL */
    const float *A_log;             /* [H] or NULL */
    float g_min, scale;             /* as kda_chunk_fwd */
    const int32_t *cu_seqlens;      /* [N + 1] device, or NULL for N sequences of T / N tokens */
    const float *initial_state;     /* [N, H, dk, dv] or NULL (zero) */
    const void *grad_o;             /* [T, H, dv] dL/do */
    const float *grad_final_state;  /* [N, H, dk, dv] dL/dS_T, or NULL (zero) */
    void *grad_q, *grad_k, *grad_z; /* [T, H, dk] outputs (grad_z is dL/dz, the gate's input) */
    void *grad_v;                   /* [T, H, dv] */
    void *grad_beta;                /* [T, H] */
    float *grad_dt_bias;            /* [H, dk], or NULL to skip */
    float *grad_A_log;              /* [H], or NULL to skip */
    float *grad_initial_state;      /* [N, H, dk, dv], or NULL to skip */
    int32_t chunk_size;             /* 64, or 0 for the default */
    int32_t gate_kind;              /* kda_gate_kind_t */
} kda_chunk_bwd_args;

/* Bytes of device scratch kda_chunk_bwd needs for one pass over all chunks (0 on invalid sizes):
 * per (chunk, head) about 0.42 MiB at d = 128 (fp32 records, L, the entering state, the leaving
 * Lambda and the chunk-local sums), independent of dtype and gate kind. */
size_t kda_chunk_bwd_workspace_size(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                    int32_t chunk_size);

/* The smallest workspace kda_chunk_bwd accepts (0 on invalid sizes).  For one sequence (N = 1)
 * longer than 16 chunks this is below kda_chunk_bwd_workspace_size: given less than the one-pass
 * size, kda_chunk_bwd processes the sequence in segments of the largest power-of-two number of
 * chunks (at least 16) whose scratch fits.  A forward sweep first stores the state entering each
 * segment; the segments then run last to first, the gradient of each one's initial state being
 * the gradient of the previous one's final state (the same recurrence as across chunks,
 * Section 5.1.2, Eq. 17), and the dt_bias and A_log gradients are the sums of the segments'
 * sums.  The results equal the one-pass results up to the rounding of those sums.  Extra
 * workspace: the entering states (64 KiB per head and segment at d = 128).  Other batches
 * (N > 1) need kda_chunk_bwd_workspace_size. */
size_t kda_chunk_bwd_workspace_size_min(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                        int32_t chunk_size);

/* Gradients must not alias the forward inputs or one another.  workspace: at least
 * kda_chunk_bwd_workspace_size_min bytes, 256-byte aligned (KDA_ERR_WORKSPACE otherwise). */
kda_status_t kda_chunk_bwd(const kda_chunk_bwd_args *args, void *workspace, size_t workspace_bytes,
                           struct CUstream_st *stream);

/* ------------------------------------------------- kda_selftest_bounded_wait
 * Not an operation of the paper: a failure-detection self-test.  Launches one CTA that waits on
 * an mbarrier nothing arrives at, through the bounded wait the tensor-core prefill and replay
 * kernels use (about one second of the global timer, then give up).  The kernel returns on its
 * own, sets KDA_ERR_DEVICE_TIMEOUT in the device error word (read it with kda_get_device_error)
 * and writes the time it waited, in ns, to *elapsed_ns (a device pointer, 8-byte aligned, or NULL).
 * The context stays usable.  Returns KDA_ERR_CUDA if there is no usable device.
 */
kda_status_t kda_selftest_bounded_wait(unsigned long long *elapsed_ns, struct CUstream_st *stream);

/* ----------------------------------------------------------- kda_output_gate
 * The output epilogue of Eq. 6 (section 2.1.1), y_t = W_o[Sigmoid(W_g x_t) * RMSNorm(o~_t)], without
 * the two projections: for every token t and head h,
 *     y[t,h,c] = Sigmoid(g[t,h,c]) * w[h,c] * o[t,h,c] / sqrt(mean_c' o[t,h,c']^2 + eps),
 * the RMSNorm taken per head over its dv value channels, g = W_g x_t given.  fp32 arithmetic.
 * Supported: dv in {32, 64, 128, 256}.  Pointers are device pointers, 16-byte aligned.
 */
typedef struct {
    int64_t T;                  /* tokens */
    int32_t H, dv;              /* heads, value channels */
    kda_dtype_t dtype;          /* dtype of o, g and y */
    const void *o;              /* [T, H, dv] recurrent output o~ */
    const void *g;              /* [T, H, dv] gate pre-activation W_g x */
    const float *norm_weight;   /* [H, dv] RMSNorm weight, or NULL (ones) */
    float eps;                  /* RMSNorm epsilon, > 0 (the report gives no value) */
    void *y;                    /* [T, H, dv] output; may alias o, must not alias g */
} kda_output_gate_args;

kda_status_t kda_output_gate(const kda_output_gate_args *args, struct CUstream_st *stream);

/* --------------------------------------------------- kda_chunk_fwd_static_ws
 * Not an operation of the paper (it has no counterpart there): the same
 * prefill as kda_chunk_fwd, for callers that cannot allocate device memory at
 * all -- for example engine plugins that receive only input and output
 * pointers while the engine owns every other byte of device memory, or code
 * that must not risk the device-wide synchronisation of cudaMalloc/cudaFree.
 * Instead of a caller workspace it uses one scratch buffer of
 * KDA_STATIC_WORKSPACE_BYTES that lives inside the library (a file-scope
 * device array, held by every GPU that loads the library until the process
 * exits).  The caller still owns and passes every input and output.
 *   - Limit: problems whose kda_chunk_fwd_workspace_size_gate() for the path
 *     they take (their gate kind; KDA_GATE_SOFTPLUS's size for a bounded gate
 *     with g_min < -5.5) exceeds KDA_STATIC_WORKSPACE_BYTES are rejected with
 *     KDA_ERR_WORKSPACE before anything is launched.  The limit depends on the
 *     gate kind and the dtype: with the bounded gate, bf16 at d = 128 needs
 *     about 73 KiB per chunk of 64 tokens per head (T = 4096 tokens with 13
 *     heads fit); the softplus gate and fp32 I/O take the fp32 path, about
 *     145 KiB per chunk and head at d = 128 (T = 4096 tokens with 7 heads fit).
 *   - Set-up: the first call on each device, made while that device is
 *     current, looks up the buffer's device address and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     A device reset (cudaDeviceReset) invalidates the kept address (and the
 *     library's device error word): do not call the library across one.
 *   - Sharing: every call on a device uses the same buffer, which keeps the
 *     last call's contents.  Calls whose GPU work overlaps in time (different
 *     streams, or different host threads) race on it and give wrong results:
 *     serialise them.
 * It allocates no device memory and calls no allocating routine. */
#define KDA_STATIC_WORKSPACE_BYTES (64u << 20)
kda_status_t kda_chunk_fwd_static_ws(const kda_chunk_args *args, struct CUstream_st *stream);

/* -------------------------------------------------------- kda_recurrent_step
 * Decode: one token per sequence, Eq. 1 applied once to each (sequence, head)
 * state in place (section 5.4.2: the recurrent state is updated in place every
 * step).  Evaluated as S' = Diag(alpha) S; e = beta (v - S'^T k);
 * S <- S' + k e^T; o = scale * (S'^T q + (k . q) e), which equals Eq. 1.
 * Supported: d_k = d_v in {64, 128}.
 */
typedef struct {
    int64_t N;                     /* sequences in this step */
    int32_t H, dk, dv;
    kda_dtype_t dtype;             /* dtype of q, k, v, z, beta and o */
    const void *q, *k, *z;         /* [N, H, dk] */
    const void *v;                 /* [N, H, dv] */
    const void *beta;              /* [N, H] */
    const float *dt_bias;          /* [H, dk] or NULL */
    const float *A_log;            /* [H] or NULL */
    float g_min, scale;
    float *state;                  /* [num_slots, H, dk, dv] fp32, read and written in place */
    const int32_t *state_indices;  /* [N] state slot of each sequence, or NULL (slot = n); the
                                      slots must be distinct (two sequences on one slot race) */
    int64_t num_slots;             /* slots in `state` (0 means N) */
    void *o;                       /* [N, H, dv] */
    int32_t gate_kind;             /* kda_gate_kind_t (0: Eq. 5) */
} kda_step_args;

kda_status_t kda_recurrent_step(const kda_step_args *args, struct CUstream_st *stream);

/* ------------------------------------------------------------------ errors */
const char *kda_status_string(kda_status_t status);

/* Waits for `stream`, then returns and clears the first device-detected error
 * (KDA_OK if none).  The word is per device and shared by all streams. */
kda_status_t kda_get_device_error(struct CUstream_st *stream);

/* The CUDA runtime error code (a cudaError_t value) behind the last
 * KDA_ERR_CUDA returned to the calling host thread, 0 if none; reading it
 * clears it. */
int32_t kda_last_cuda_error(void);

int kda_abi_version(void);

/* ------------------------------------------------------------- debug checks
 * Not an operation of the paper: optional checks for debugging a model.  With KDA_CHECK_FINITE set,
 * every entry point that writes results (kda_gate, kda_chunk_fwd and kda_chunk_fwd_static_ws,
 * kda_recurrent_step, kda_recurrent_replay, kda_output_gate, kda_chunk_bwd) launches one more pass
 * over what it wrote (outputs, final or updated states, gradients) that sets KDA_ERR_NUMERIC in the
 * device error word (kda_get_device_error) when any value is NaN or infinite.  The pass reads those
 * results once more from HBM.  Index checks need no switch: cu_seqlens contents, state indices and
 * replay counts are always checked on the device.  Process-wide; 0 (the default) turns the checks
 * off.  KDA_ERR_INVALID_ARG for an unknown flag. */
#define KDA_CHECK_FINITE 1
kda_status_t kda_set_debug_checks(int32_t flags);

/* ------------------------------------------------------------ instrumentation
 * Optional per-kernel timing.  While set (n_events > 0), kda_chunk_fwd records
 * events[0] on its stream before its first kernel and events[i] right after its
 * i-th kernel launch, for i < n_events; kda_recurrent_step records events[0]
 * before and events[1] after its kernel.  `events` are cudaEvent_t handles
 * created by the caller (timing enabled); the array is copied.  Pass
 * (NULL, 0) to stop.  Process-wide setting: set it only while one thread calls
 * into the library.  Returns the number of kernels kda_chunk_fwd launches for
 * the given problem when queried with kda_chunk_fwd_kernel_count(). */
kda_status_t kda_set_profile_events(void *const *events, int32_t n_events);
int32_t kda_chunk_fwd_kernel_count(const kda_chunk_args *args);

/* The schedule kda_chunk_fwd picks for these arguments (host only: reads the
 * sizes, dtype and cu_seqlens_host, launches nothing).  out (caller-owned, 4
 * entries): out[0] = 1 for the fused launch (intra-chunk transform and output
 * pass in one cooperative kernel, one CTA per chain), 2 for the chain-team
 * launch (one cooperative kernel of teams, each a chain CTA that runs its chains
 * in turn and out[1] CTAs producing their packets just ahead of it), else 0;
 * out[1] = chunks at the start of every sequence that its own output-pass CTAs
 * produce in the fused launch, or producers per team; out[2] =
 * segment length in chunks of the split-sequence state pass (the Kimi K3
 * report, section 5.1.2, Eq. 17), 0 when the pass does not run; out[3] =
 * kernels launched.  KDA_ERR_INVALID_ARG on NULL pointers or invalid sizes. */
kda_status_t kda_chunk_fwd_schedule(const kda_chunk_args *args, int64_t *out);

/* Not an operation of the paper: the schedule of the bf16 d = 128 tensor-core prefill, for tests and
 * measurements.  KDA_SCHEDULE_AUTO (the default) lets the library's latency model choose; the others
 * force the separate kernels, the fused launch or the chain-team launch when the problem is eligible
 * for it (fused: sequences x heads + 16 <= SMs; team: at most 159 sequences), else the model's choice
 * among what remains.  The model never picks the chain-team launch: on a GB300 it measured 2-4x
 * slower than the separate kernels or the fused launch on every workload tried.  Every schedule computes the same result.  Process-wide; applies to later
 * calls of kda_chunk_fwd, its workspace size and kda_chunk_fwd_schedule alike.  KDA_ERR_INVALID_ARG
 * for an unknown mode. */
#define KDA_SCHEDULE_AUTO 0
#define KDA_SCHEDULE_SEPARATE 1
#define KDA_SCHEDULE_FUSED 2
#define KDA_SCHEDULE_TEAM 3
kda_status_t kda_set_chunk_schedule(int32_t mode);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
