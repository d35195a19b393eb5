// Chunk planning for kda_chunk_fwd: workspace layout (host) and the
// per-sequence chunk offsets (device).
//
// Chunks of C tokens start at each sequence's first token (the last chunk of a
// sequence may be shorter).  Chunk slots are numbered sequence by sequence:
// sequence n owns slots [chunk_start[n], chunk_start[n + 1]).  The number of
// slots is bounded on the host without reading cu_seqlens:
//     sum_n ceil(len_n / C) <= floor((T + N (C - 1)) / C),
// so kernels are launched over that bound and slots past chunk_start[N] exit.
#include "kda_common.cuh"
#include "kda_internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>

namespace kda {

__global__ void __launch_bounds__(1024)
chunk_plan_kernel(const int32_t *__restrict__ cu, int64_t T, int N, int C,
                  int32_t *__restrict__ chunk_start, int64_t seg_len, int32_t *__restrict__ seg_start,
                  int32_t *__restrict__ unit_seg, int *__restrict__ unit_ctr, int *err) {
    constexpr int MAX_SORT = 4096;  // segments ordered by length; more are taken in index order
    __shared__ int s_cnt[MAX_SORT];
    __shared__ int s_bad;
    __shared__ int s_warp[32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) { s_bad = 0; s_carry = 0; }
    __syncthreads();
    if (cu) {
        for (int n = tid; n <= N; n += blockDim.x) {
            const int64_t x = cu[n];
            bool bad = (n == 0 && x != 0) || (n == N && x != T) || (n > 0 && x < (int64_t)cu[n - 1]);
            if (bad) atomicOr(&s_bad, 1);
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) set_error(err, KDA_ERR_BAD_SEQLENS);
        for (int n = tid; n <= N; n += blockDim.x) {
            chunk_start[n] = 0;  // no chunk runs
            if (seg_start) seg_start[n] = 0;
        }
        return;
    }
    const int64_t len_eq = cu ? 0 : T / N;
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        int cnt = 0;
        if (n < N) {
            const int64_t len = cu ? (int64_t)cu[n + 1] - cu[n] : len_eq;
            cnt = (int)((len + C - 1) / C);
        }
        int x = cnt;  // inclusive scan across the block
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0) + s_carry;
        if (n < N) chunk_start[n + 1] = incl;
        __syncthreads();
        if (tid == blockDim.x - 1) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_start[0] = 0;
    if (!seg_start) return;
    // segments per sequence: max(1, ceil(chunks / seg_len)) (an empty sequence keeps one segment,
    // which writes its final state)
    __syncthreads();
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        int cnt = 0;
        if (n < N) {
            const int64_t nc = (int64_t)chunk_start[n + 1] - chunk_start[n];
            cnt = (int)max((int64_t)1, (nc + seg_len - 1) / seg_len);
        }
        int x = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0) + s_carry;
        if (n < N) seg_start[n + 1] = incl;
        __syncthreads();
        if (tid == blockDim.x - 1) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) seg_start[0] = 0;
    if (!unit_seg) return;
    // the output pass takes segments longest first (fewer short chains left for the tail), from a
    // counter this kernel resets
    __syncthreads();
    if (tid == 0) *unit_ctr = 0;
    const int S = seg_start[N];
    if (S > MAX_SORT) {
        for (int g = tid; g < S; g += blockDim.x) unit_seg[g] = g;
        return;
    }
    for (int n = tid; n < N; n += blockDim.x) {
        const int nc = chunk_start[n + 1] - chunk_start[n];
        for (int g = seg_start[n]; g < seg_start[n + 1]; ++g) {
            const int64_t left = (int64_t)nc - (int64_t)(g - seg_start[n]) * seg_len;
            s_cnt[g] = (int)max((int64_t)0, min(seg_len, left));
        }
    }
    __syncthreads();
    for (int g = tid; g < S; g += blockDim.x) {  // rank by (chunks descending, index ascending)
        const int c = s_cnt[g];
        int r = 0;
        for (int x = 0; x < S; ++x) r += (s_cnt[x] > c || (s_cnt[x] == c && x < g)) ? 1 : 0;
        unit_seg[r] = g;
    }
}

}  // namespace kda

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Schedule of the tensor-core path, from a latency model of its kernels (microseconds, one CTA per
// SM): an intra-chunk item costs T_ITEM, plus T_COLD for the first item of a CTA; a step of the
// output pass T_CHAIN, of a segment summary T_SUM, of the fold T_FOLD; T_LAUNCH per kernel boundary.
// Three schedules:
//  - separate kernels, one segment per sequence;
//  - separate kernels with the split-sequence state pass (segments of L chunks);
//  - fused: chains (one per sequence and head) and intra-chunk producers share one launch; each
//    chain first produces its own first kpre chunks, the producers the rest.
// Uses per-sequence lengths when the host copy of cu_seqlens is given.
constexpr double T_ITEM = 6.5, T_COLD = 13.5, T_CHAIN = 1.15, T_SUM = 2.3, T_FOLD = 1.8, T_LAUNCH = 4.0;
constexpr double T_CHAIN_START = 3.0;      // a chain CTA switching to its next chain (team schedule)
constexpr double TEAM_MAX_CHAINS_HOST = 512;  // chains per team the producers' table holds

struct tc_schedule {
    int64_t seg_len;  // 1 << 30: no split
    bool fused;
    int kpre;
    bool team;
    int teams, team_k;
};

static tc_schedule choose_schedule(int64_t T, int64_t N, int H, int C, const int32_t *cu_host, int sms,
                                   int force = KDA_SCHEDULE_AUTO) {
    tc_schedule r{(int64_t)1 << 30, false, 0, false, 0, 0};
    if (T == 0) return r;
    int64_t total = 0, longest = 0;
    auto chunks_of = [&](int64_t n) -> int64_t {
        const int64_t len = cu_host ? (int64_t)cu_host[n + 1] - cu_host[n] : T / N;
        return (len + C - 1) / C;
    };
    for (int64_t n = 0; n < N; ++n) {
        const int64_t c = chunks_of(n);
        total += c;
        longest = c > longest ? c : longest;
    }
    auto waves = [&](double ctas, double width) { return std::ceil(ctas / width); };
    const double items = (double)total * H;
    const double intra = T_COLD + waves(items, sms) * T_ITEM;
    // unsplit output pass: the longest chain, or the chains' total over the SMs
    const double unsplit = (double)longest > items / sms ? (double)longest : items / sms;
    double best = intra + unsplit * T_CHAIN + 2 * T_LAUNCH;
    if (force == KDA_SCHEDULE_SEPARATE) return r;
    if (force == KDA_SCHEDULE_FUSED || force == KDA_SCHEDULE_TEAM) best = 1e300;  // any eligible one of that kind
    for (int64_t L = 8; L <= (1 << 14) && force == KDA_SCHEDULE_AUTO; L *= 2) {
        if (L >= longest) break;
        int64_t segs = 0, segs_sum = 0, max_nseg = 0;
        for (int64_t n = 0; n < N; ++n) {
            const int64_t c = chunks_of(n);
            const int64_t ns = c > 0 ? (c + L - 1) / L : 1;
            segs += ns;
            segs_sum += ns - 1;
            max_nseg = ns > max_nseg ? ns : max_nseg;
        }
        const double steps = T_SUM * L * waves((double)segs_sum * H, sms) + T_FOLD * (max_nseg - 1) +
                             T_CHAIN * L * waves((double)segs * H, sms);
        const double cost = intra + steps + 4 * T_LAUNCH;
        if (cost < 0.85 * best) {  // split only for a clear gain
            best = cost;
            r.seg_len = L;
        }
    }
    const int64_t n_chain = N * H;
    if (n_chain + 16 <= sms && N <= KDA_FUSED_MAX_SEQS && force != KDA_SCHEDULE_TEAM) {
        const double producers = (double)(sms - n_chain);
        for (int kp = 0; kp <= 8; ++kp) {
            double items_p = 0;
            for (int64_t n = 0; n < N; ++n) {
                const int64_t c = chunks_of(n) - kp;
                items_p += c > 0 ? (double)c * H : 0.0;
            }
            const double pm = items_p > 0 ? T_COLD + waves(items_p, producers) * T_ITEM : 0.0;
            const double first = T_COLD + (kp > 0 ? (double)(kp < longest ? kp : longest) : 1.0) * T_ITEM;
            const double chain_end = std::max(first + (double)longest * T_CHAIN, pm + 2 * T_CHAIN);
            const double cost = std::max(pm, chain_end) + T_LAUNCH;
            if (cost < best) {
                best = cost;
                r.fused = true;
                r.kpre = kp;
                r.seg_len = (int64_t)1 << 30;
            }
        }
    }
    // chain teams: teams of one chain CTA and k producers; the chains, dealt longest first in snake
    // order, give every team about the same number of chunk steps.  Only on request: measured on GB300
    // (T=4096 x 32 heads, 32 x 4.3K-token varlen batch, T=1M x 32 heads) it is 2-4x slower than the
    // other schedules, its chain steps waiting on packets that left L2 (see kda_set_chunk_schedule).
    if (N <= KDA_FUSED_MAX_SEQS && force == KDA_SCHEDULE_TEAM &&
        (double)n_chain <= (double)(sms / 2) * TEAM_MAX_CHAINS_HOST) {
        for (int k = 1; k <= 8; ++k) {
            const int teams = sms / (k + 1);
            if (teams < 1 || teams > KDA_CTR_MAX || (double)n_chain > (double)teams * TEAM_MAX_CHAINS_HOST) continue;
            const double per_team = items / teams;  // chunk steps (= packets) per team
            const double chain = std::max(per_team, (double)longest) * T_CHAIN +
                                 std::ceil((double)n_chain / teams) * T_CHAIN_START;
            const double prod = per_team * T_ITEM / k;
            const double cost = T_COLD + std::max(chain, prod) + T_LAUNCH;
            if (cost < best) {
                best = cost;
                r.team = true;
                r.teams = teams;
                r.team_k = k;
                r.fused = false;
                r.kpre = 0;
                r.seg_len = (int64_t)1 << 30;
            }
        }
    }
    return r;
}

namespace {
std::atomic<int> g_schedule_override{0};  // kda_set_chunk_schedule
}

int kda_chunk_schedule_override() { return g_schedule_override.load(std::memory_order_relaxed); }

extern "C" kda_status_t kda_set_chunk_schedule(int32_t mode) {
    if (mode < KDA_SCHEDULE_AUTO || mode > KDA_SCHEDULE_TEAM) return KDA_ERR_INVALID_ARG;
    g_schedule_override.store(mode, std::memory_order_relaxed);
    return KDA_OK;
}

bool kda_make_chunk_plan(int64_t T, int64_t N, int H, int dk, int dv, kda_dtype_t dtype, int C,
                         kda_chunk_plan *p, const int32_t *cu_seqlens_host, int gate_kind,
                         bool force_fp32_path) {
    if (T < 0 || N < 1 || H < 1 || C < 1) return false;
    p->T = T; p->N = N; p->H = H; p->dk = dk; p->dv = dv; p->C = C;
    p->max_chunks = (T + N * (int64_t)(C - 1)) / C;
    // bf16 with d_k = d_v = 128 and the bounded gate runs on the tensor cores; everything else on
    // the fp32 CUDA-core path, and so does an empty batch (T = 0: no tiles to map, only the states
    // to pass through)
    p->path = (T > 0 && dtype == KDA_BF16 && dk == 128 && dv == 128 && C == 64 &&
               gate_kind == KDA_GATE_LOWER_BOUND && !force_fp32_path) ? 1 : 0;
    if (p->path == 1) {
        p->record_bytes = kda_tc_packet_stride();  // bf16 operand images + gamma^C
    } else {
        // fp32 CUDA-core records: W, Q^, K~ [C, dk]; U [C, dv]; A [C, C]; gamma^C [dk]
        p->record_bytes = align_up(sizeof(float) * ((size_t)C * (3 * dk + dv) + (size_t)C * C + dk), 256);
    }
    p->off_chunk_start = 0;
    p->off_records = align_up(sizeof(int32_t) * (size_t)(N + 1), 256);
    size_t end = p->off_records + p->record_bytes * (size_t)p->max_chunks * (size_t)H;
    p->split = 0;
    p->fused = 0;
    p->kpre = 0;
    p->team = 0;
    p->teams = p->team_k = p->team_window = 0;
    p->epi_fused = 0;
    p->seg_len = (int64_t)1 << 30;
    p->max_segs = N;
    if (p->path == 1) {
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
        const tc_schedule sch = choose_schedule(T, N, H, C, cu_seqlens_host, sms, kda_chunk_schedule_override());
        p->seg_len = sch.seg_len;
        p->fused = sch.fused ? 1 : 0;
        p->kpre = sch.kpre;
        p->team = sch.team ? 1 : 0;
        p->teams = sch.teams;
        p->team_k = sch.team_k;
        p->team_window = 6;  // own items a producer may run ahead of its chain
        // the output epilogue inside the output pass adds ~2.8K cycles of output-warp work per chunk: cheaper
        // than its own pass over o where chains run as separate kernels (a 32 x 4.3K-token batch: +0.39 ms
        // against +0.62 ms), dearer in the one-launch schedule, whose chains bound the launch (T = 256K x 32
        // heads: +56 % against +16 %)
        p->epi_fused = p->fused ? 0 : 1;
        p->split = p->seg_len < ((int64_t)1 << 30) ? 1 : 0;
        p->max_segs = p->split ? p->max_chunks / p->seg_len + N : N;
    }
    p->off_seg_start = align_up(end, 256);
    end = p->off_seg_start + sizeof(int32_t) * (size_t)(N + 1);
    p->off_seg_sum = align_up(end, 1024);
    p->off_seg_in = p->off_seg_sum;
    if (p->split) {
        p->off_seg_in = p->off_seg_sum + (size_t)p->max_segs * H * 2 * 128 * 128 * sizeof(float);
        end = p->off_seg_in + (size_t)p->max_segs * H * 128 * 128 * sizeof(float);
    }
    p->off_flags = align_up(end, 256);
    end = p->off_flags + sizeof(uint64_t) * (size_t)p->max_chunks * (size_t)H;
    p->off_consumed = align_up(end, 256);
    if (p->team) end = p->off_consumed + sizeof(uint64_t) * (size_t)p->max_chunks * (size_t)H;
    p->off_ctr = align_up(end, 256);
    if (p->path == 1) end = p->off_ctr + sizeof(uint64_t) * KDA_CTR_STRIDE * KDA_CTR_MAX;
    p->off_unit = align_up(end, 256);
    if (p->path == 1) end = p->off_unit + sizeof(int32_t) * (size_t)p->max_segs;
    p->total_bytes = align_up(end, 256);
    return true;
}

kda_status_t kda_launch_chunk_plan(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                   cudaStream_t stream) {
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    int32_t *chunk_start = (int32_t *)((char *)ws + p.off_chunk_start);
    int32_t *seg_start = p.path == 1 ? (int32_t *)((char *)ws + p.off_seg_start) : nullptr;
    int32_t *unit_seg = p.path == 1 ? (int32_t *)((char *)ws + p.off_unit) : nullptr;
    int *unit_ctr = p.path == 1 ? (int *)((char *)ws + p.off_ctr + sizeof(uint64_t) * KDA_CTR_STRIDE) : nullptr;
    kda::chunk_plan_kernel<<<1, 1024, 0, stream>>>(a->cu_seqlens, a->T, (int)a->N, p.C, chunk_start,
                                                    p.seg_len, seg_start, unit_seg, unit_ctr, err);
    return kda_cuda_status(cudaGetLastError());
}
