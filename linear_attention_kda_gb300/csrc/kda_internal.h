// Internal launchers behind the C ABI (host side).  Arguments are validated by
// kda_api.cu before any of these is called.
#pragma once
#include <cuda_runtime.h>

#include "../../include/kda.h"

// Records the i-th profiling event on `stream` when instrumentation is set.
void kda_profile_mark(int i, cudaStream_t stream);
// KDA_OK for cudaSuccess; otherwise records the code for kda_last_cuda_error() and returns KDA_ERR_CUDA.
kda_status_t kda_cuda_status(cudaError_t e);

// Debug checks (kda_set_debug_checks): the flags in force, and the scan that sets KDA_ERR_NUMERIC in
// the device error word when [p, p + n) holds a NaN or an infinity (p 16-byte aligned).
int32_t kda_debug_flags();
kda_status_t kda_check_finite(const void *p, int64_t n, kda_dtype_t dtype, cudaStream_t stream);

kda_status_t kda_launch_gate(const kda_gate_args *a, cudaStream_t stream);
kda_status_t kda_launch_output_gate(const kda_output_gate_args *a, cudaStream_t stream);
kda_status_t kda_launch_decode(const kda_step_args *a, cudaStream_t stream);
kda_status_t kda_launch_replay(const kda_replay_args *a, cudaStream_t stream);

// Chunked prefill.  Workspace layout is owned by kda_chunk_plan.cu.
constexpr int KDA_FUSED_MAX_SEQS = 159;  // sequences the fused schedule's producer item map holds
constexpr int KDA_CTR_MAX = 128;         // producer item counters (one per chain team, or one)
constexpr int KDA_CTR_STRIDE = 16;       // uint64 words between counters (one 128-byte line each)
struct kda_chunk_plan {
    int64_t T, N;
    int H, dk, dv, C;
    int64_t max_chunks;    // upper bound on chunks over all sequences
    int path;              // 0 = fp32 CUDA-core path, 1 = tensor-core path
    size_t off_chunk_start;  // int32 [N + 1]: first chunk slot of each sequence
    size_t off_records;      // per (chunk slot, head) intra-chunk records
    size_t record_bytes;
    // Split-sequence state pass (tensor-core path): sequences are cut into segments of seg_len
    // chunks; every segment but the last of its sequence gets a summary (S~, M) with
    // S_out = M S_in + S~, the summaries are folded in order, and each segment then runs from its
    // true entering state.  seg_len >= max chunks per sequence means one segment per sequence.
    int split;               // 1 if the segment summary and fold passes run
    int64_t seg_len;         // chunks per segment
    int64_t max_segs;        // upper bound on segments over all sequences
    size_t off_seg_start;    // int32 [N + 1]: first segment of each sequence
    size_t off_seg_sum;      // per (segment, head), 128 KB: S~ [128][128] fp32 (lane-major), then M as bf16
                             // high and low operand images (32 KB each)
    size_t off_seg_in;       // per (segment, head): entering state S [128][128] fp32 (lane-major)
    // Fused launch (tensor-core path, no split): the output pass of every (sequence, head) and the
    // intra-chunk work run concurrently in one cooperative launch (no planning kernel); packets are
    // published through 64-bit epoch flags, one per (chunk slot, head).
    int fused;               // (at most KDA_FUSED_MAX_SEQS sequences)
    int kpre;                // fused: chunks at the start of every sequence that its chains produce themselves
    // Chain teams (tensor-core path, many chains): one cooperative launch of `teams` teams, each a
    // chain CTA and team_k producer CTAs; producers run at most team_window of their own items ahead.
    int team;                // 1 if the team schedule runs (then fused = 0)
    // The output epilogue (out_gate) runs inside the output pass instead of as its own pass over o.  Not
    // for the fused launch, whose chains bound the launch.
    int epi_fused;
    int teams, team_k, team_window;
    size_t off_flags;
    size_t off_consumed;     // team schedule: per (chunk slot, head), the epoch once its chain has started on it
    size_t off_ctr;          // tensor-core path: item counters of the producers (KDA_CTR_MAX, 128 bytes apart)
    size_t off_unit;         // tensor-core path: int32 [max_segs] segments in the order the output pass takes them
    size_t total_bytes;
};

// The schedule forced by kda_set_chunk_schedule (KDA_SCHEDULE_AUTO: the latency model chooses).
int kda_chunk_schedule_override();

// gate_kind KDA_GATE_SOFTPLUS always takes the fp32 CUDA-core path (its in-chunk decays are not
// bounded, so the tensor-core operand images could overflow).
bool kda_make_chunk_plan(int64_t T, int64_t N, int H, int dk, int dv, kda_dtype_t dtype, int C,
                         kda_chunk_plan *plan, const int32_t *cu_seqlens_host = nullptr, int gate_kind = 0,
                         bool force_fp32_path = false);
kda_status_t kda_launch_chunk_simt(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                   cudaStream_t stream);
kda_status_t kda_launch_chunk_tc(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                 cudaStream_t stream);
// The fp32 forward again, for the backward pass: records as kda_launch_chunk_simt, plus L per
// (chunk slot, head) [C][C] into Lout and the state entering each chunk slot [dk][dv] into ckpt;
// o is written only when a->o is set.
// The bf16 tensor-core prefill scales the rows and keys of a 64-token chunk by e^{G_r - G_p} against
// references p at most 16 tokens away, so every such exponent is at most 16 |g_min| in size: inside
// fp32 / bf16 range (e^88.7) for g_min >= -5.5 (the report uses -5).  A bounded gate with a lower g_min
// runs on the fp32 path, whose decays are exp(G_r - G_i) <= 1 for every gate.
constexpr float KDA_TC_MIN_G_MIN = -5.5f;
inline bool kda_gate_needs_fp32_path(int gate_kind, float g_min) {
    return gate_kind == KDA_GATE_LOWER_BOUND && !(g_min >= KDA_TC_MIN_G_MIN);
}
// The gate kind whose kda_chunk_fwd_workspace_size_gate fits a call: the softplus gate's (the fp32
// path's) for a bounded gate below KDA_TC_MIN_G_MIN.
inline int kda_workspace_gate(int gate_kind, float g_min) {
    return kda_gate_needs_fp32_path(gate_kind, g_min) ? (int)KDA_GATE_SOFTPLUS : gate_kind;
}
// The backward pass's forward chain (checkpoints) on the tensor cores: launched and true when the problem
// allows it (bf16, d_k = d_v = 128, no outputs, checkpoints requested), else false.
bool kda_launch_chain_ckpt_tc(const kda_chunk_args *a, const int32_t *chunk_start, const char *records,
                              size_t rec_bytes, float *ckpt, cudaStream_t stream);
kda_status_t kda_launch_chunk_simt_recompute(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                             float *Lout, float *ckpt, cudaStream_t stream);
size_t kda_tc_packet_stride();  // bytes per (chunk, head) packet of the tensor-core path

// Backward pass of the chunked prefill (kda_chunk_bwd.cu): scratch bytes for these sizes (0 if
// invalid) and the launcher (arguments validated by kda_api.cu).
size_t kda_chunk_bwd_layout_bytes(int64_t T, int64_t N, int H, int dk, int dv);
// The smallest workspace kda_launch_chunk_bwd accepts: a single sequence longer than 16 chunks runs in
// segments when the whole pass does not fit (segments of 16 chunks at this size).
size_t kda_chunk_bwd_min_layout_bytes(int64_t T, int64_t N, int H, int dk, int dv);
kda_status_t kda_launch_chunk_bwd(const kda_chunk_bwd_args *a, void *ws, size_t ws_bytes, cudaStream_t stream);
