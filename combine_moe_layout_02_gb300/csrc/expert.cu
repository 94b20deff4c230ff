// expert.cu -- receive rows of the expert-major layout (moe_notify_expert).
//
// "HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 3.6 (InputToShare): each
// (token, k) slot goes to row dstExpertOffset + curExpertCnt of its expert on
// the destination rank, so the rows of one expert are contiguous and in
// (token, k) order, ready for a grouped expert GEMM. Expert l of rank d starts
// at recv_expert_offset[d][l] (moe_notify: the exclusive scan of the counts
// rounded up to expert_alignment, "internode.cu" section 1).
//
//   slot_row[g][k] = recv_expert_offset[e] + #(slots of expert e before (g, k))
//   expert_part_base[d] = sum over d' < d of sum_l num_recv_tokens_per_expert[d'][l]
//
// Three launches over "chunks" of kChunkTokens consecutive tokens, one warp per
// chunk. Inside a warp the K slots of 32 / K consecutive tokens sit on the
// lanes in (token, k) order, so __match_any_sync groups equal experts and the
// popcount of the lower lanes of a group is the slot's rank among them.
//  1. count: per-chunk expert histograms (warp-private shared counters, one
//     writer per address per step) into scratch [chunks][E];
//  2. scan: one warp per expert turns its column into exclusive chunk bases
//     plus recv_expert_offset (in place); warp 0 of the last block also scans
//     the rank totals into expert_part_base;
//  3. rows: each chunk's warp starts its counters at those bases and assigns
//     every slot its row in order.
// Integer counts in a fixed order: deterministic, no atomics.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kChunkTokens = 64;
constexpr int kThreads = 256;

struct ExpertPlan {
    int64_t chunks;
    int wpb;           // warps (chunks) per block, bounded by E counters in shared memory
    int64_t blocks;    // blocks of the chunk kernels
    size_t smem;       // wpb * E * 4
    int64_t scratch_bytes;
};

ExpertPlan expert_plan(const moe_shape& s) {
    ExpertPlan p;
    p.chunks = ceil_div(s.S, kChunkTokens);
    int wpb = static_cast<int>((64 * 1024) / (static_cast<int64_t>(s.E) * 4));
    p.wpb = wpb < 1 ? 1 : (wpb > kThreads / 32 ? kThreads / 32 : wpb);
    p.blocks = ceil_div(p.chunks, p.wpb);
    p.smem = static_cast<size_t>(p.wpb) * s.E * 4;
    p.scratch_bytes = round_up(p.chunks * s.E * 4, 256);
    return p;
}

// Walk one chunk's slots in (token, k) order. For each step f(step_base_slot,
// e, group) is called on every lane: e is the lane's expert (-1 for a masked,
// invalid or idle lane) and group its __match_any_sync mask.
template <typename F>
__device__ __forceinline__ void walk_chunk(const int32_t* __restrict__ topk_idx, int64_t g0, int64_t g1,
                                           int K, int E, int lane, F&& f) {
    const int tps = 32 / K;                 // tokens per step
    const int used = tps * K;               // lanes carrying a slot
    for (int64_t gs = g0; gs < g1; gs += tps) {
        const int64_t g = gs + lane / K;
        const int k = lane % K;
        int32_t e = -1;
        if (lane < used && g < g1) {
            e = __ldg(topk_idx + g * K + k);
            if (e < 0 || e >= E) e = -1;
        }
        const uint32_t grp = __match_any_sync(0xffffffffu, e);
        f(g, k, e, grp);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kThreads)
expert_count_kernel(int32_t E, int32_t K, int64_t S, int64_t chunks, const int32_t* __restrict__ topk_idx,
                    int32_t* __restrict__ ecount) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) int32_t hist_all[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    if (chunk >= chunks) return;
    int32_t* hist = hist_all + warp * E;
    for (int e = lane; e < E; e += 32) hist[e] = 0;
    __syncwarp();
    const int64_t g0 = chunk * kChunkTokens;
    const int64_t g1 = g0 + kChunkTokens < S ? g0 + kChunkTokens : S;
    walk_chunk(topk_idx, g0, g1, K, E, lane, [&](int64_t, int, int32_t e, uint32_t grp) {
        if (e >= 0 && lane == 31 - __clz(grp)) hist[e] += __popc(grp);
    });
    for (int e = lane; e < E; e += 32) ecount[chunk * E + e] = hist[e];
}

__global__ void __launch_bounds__(kThreads)
expert_scan_kernel(int32_t P, int32_t E, int64_t chunks, const int32_t* __restrict__ reo,
                   const int32_t* __restrict__ nrtpe, int32_t* __restrict__ ecount,
                   int64_t* __restrict__ expert_part_base) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw < E) {
        const int64_t e = gw;
        int32_t carry = __ldg(reo + e);
        for (int64_t c0 = 0; c0 < chunks; c0 += 32) {
            const int64_t c = c0 + lane;
            const int32_t v = c < chunks ? ecount[c * E + e] : 0;
            int32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (c < chunks) ecount[c * E + e] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    } else if (gw == E) {
        const int epr = E / P;
        int64_t run = 0;
        for (int d0 = 0; d0 < P; d0 += 32) {
            const int d = d0 + lane;
            int64_t v = 0;
            if (d < P)
                for (int l = 0; l < epr; ++l) v += __ldg(nrtpe + static_cast<int64_t>(d) * epr + l);
            int64_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (d < P) expert_part_base[d] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) expert_part_base[P] = run;
    }
}

__global__ void __launch_bounds__(kThreads)
expert_rows_kernel(int32_t E, int32_t K, int64_t S, int64_t chunks, const int32_t* __restrict__ topk_idx,
                   const int32_t* __restrict__ ebase, int32_t* __restrict__ slot_row) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) int32_t hist_all[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    if (chunk >= chunks) return;
    int32_t* next = hist_all + warp * E;
    for (int e = lane; e < E; e += 32) next[e] = __ldg(ebase + chunk * E + e);
    __syncwarp();
    const int64_t g0 = chunk * kChunkTokens;
    const int64_t g1 = g0 + kChunkTokens < S ? g0 + kChunkTokens : S;
    walk_chunk(topk_idx, g0, g1, K, E, lane, [&](int64_t g, int k, int32_t e, uint32_t grp) {
        if (g < g1 && lane < (32 / K) * K) {
            int32_t row = -1;
            if (e >= 0) row = next[e] + __popc(grp & lanemask_lt());
            slot_row[g * K + k] = row;
        }
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(grp)) next[e] += __popc(grp);
    });
}

}  // namespace

int64_t notify_expert_scratch_bytes(const moe_shape& s) { return expert_plan(s).scratch_bytes; }

cudaError_t launch_notify_expert(const moe_shape& s, const int32_t* topk_idx, const int32_t* nrtpe,
                                 const int32_t* reo, int32_t* slot_row, int64_t* expert_part_base,
                                 void* scratch, cudaStream_t stream) {
    const ExpertPlan p = expert_plan(s);
    int32_t* ecount = static_cast<int32_t*>(scratch);
    cudaError_t e = cudaSuccess;
    if (p.chunks > 0) {
        e = prepare_kernel(reinterpret_cast<const void*>(expert_count_kernel), p.smem, p.wpb * 32, nullptr);
        if (e != cudaSuccess) return e;
        e = prepare_kernel(reinterpret_cast<const void*>(expert_rows_kernel), p.smem, p.wpb * 32, nullptr);
        if (e != cudaSuccess) return e;
        e = launch_pdl(expert_count_kernel, static_cast<unsigned>(p.blocks), p.wpb * 32, p.smem, stream, s.E,
                       s.K, static_cast<int64_t>(s.S), p.chunks, topk_idx, ecount);
        if (e != cudaSuccess) return e;
    }
    const int64_t scan_warps = static_cast<int64_t>(s.E) + 1;
    e = launch_pdl(expert_scan_kernel, static_cast<unsigned>(ceil_div(scan_warps, kThreads / 32)), kThreads, 0,
                   stream, s.P, s.E, p.chunks, reo, nrtpe, ecount, expert_part_base);
    if (e != cudaSuccess || p.chunks == 0) return e;
    return launch_pdl(expert_rows_kernel, static_cast<unsigned>(p.blocks), p.wpb * 32, p.smem, stream, s.E, s.K,
                      static_cast<int64_t>(s.S), p.chunks, topk_idx, static_cast<const int32_t*>(ecount),
                      slot_row);
}

}  // namespace moe
