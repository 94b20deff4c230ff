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
// Three launches over "chunks" of kChunkTokens consecutive tokens. A chunk's
// slots are contiguous in topk_idx ([S, K] row-major), so one warp loads all
// of them at once, 32 consecutive slots per step, lanes in (token, k) order.
//  1. count: per-chunk expert histograms (shared-memory integer atomics) into
//     scratch, expert-major: ecount[e][chunk];
//  2. scan: one warp per expert turns its contiguous column into the chunks'
//     first rows (16-byte loads, one warp scan per 512 chunks), starting at
//     recv_expert_offset, written chunk-major: ebase[chunk][e]; one more warp
//     scans the rank totals into expert_part_base;
//  3. rows: each chunk's warp starts its counters at those bases and ranks
//     every slot among the step's slots of the same expert
//     (__match_any_sync), in (token, k) order.
// Integer counts: the result does not depend on the order of the atomics.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kChunkTokens = 32;
constexpr int kThreads = 256;
constexpr int kMaxSteps = kChunkTokens * 16 / 32;  // slots per chunk / 32, for K <= 16
constexpr int kSeg = 16;                            // chunks per lane per scan block

struct ExpertPlan {
    int64_t chunks, chunks_pad;  // chunk count; expert-major row stride (multiple of 4)
    int wpb;                     // warps (chunks) per block, bounded by E counters in shared memory
    int64_t blocks;              // blocks of the chunk kernels
    size_t smem;                 // wpb * E * 4
    int64_t ebase_off, scratch_bytes;
};

ExpertPlan expert_plan(const moe_shape& s) {
    ExpertPlan p;
    p.chunks = ceil_div(s.S, kChunkTokens);
    p.chunks_pad = round_up(p.chunks, 4);
    int wpb = static_cast<int>((64 * 1024) / (static_cast<int64_t>(s.E) * 4));
    p.wpb = wpb < 1 ? 1 : (wpb > kThreads / 32 ? kThreads / 32 : wpb);
    p.blocks = ceil_div(p.chunks, p.wpb);
    p.smem = static_cast<size_t>(p.wpb) * s.E * 4;
    p.ebase_off = round_up(static_cast<int64_t>(s.E) * p.chunks_pad * 4, 256);
    p.scratch_bytes = p.ebase_off + round_up(p.chunks * s.E * 4, 256);
    return p;
}

// The chunk's slots, 32 per step: lane `lane` of step st holds slot
// f = 32 * st + lane of the chunk ((token, k) order), or -1 beyond the chunk
// or for a masked / out-of-range id.
__device__ __forceinline__ void load_chunk(const int32_t* __restrict__ topk_idx, int64_t f0, int nslots, int E,
                                           int lane, int32_t (&ids)[kMaxSteps]) {
#pragma unroll
    for (int st = 0; st < kMaxSteps; ++st) {
        const int f = st * 32 + lane;
        int32_t e = -1;
        if (f < nslots) {
            e = __ldg(topk_idx + f0 + f);
            if (e < 0 || e >= E) e = -1;
        }
        ids[st] = e;
    }
}

__global__ void __launch_bounds__(kThreads)
expert_count_kernel(int32_t E, int32_t K, int64_t S, int64_t chunks, int64_t chunks_pad,
                    const int32_t* __restrict__ topk_idx, int32_t* __restrict__ ecount) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) int32_t hist_all[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t chunk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    if (chunk >= chunks) return;
    int32_t* hist = hist_all + warp * E;
    const int64_t g0 = chunk * kChunkTokens;
    const int64_t g1 = g0 + kChunkTokens < S ? g0 + kChunkTokens : S;
    const int nslots = static_cast<int>((g1 - g0) * K);
    int32_t ids[kMaxSteps];
    load_chunk(topk_idx, g0 * K, nslots, E, lane, ids);
    for (int e = lane; e < E; e += 32) hist[e] = 0;
    __syncwarp();
#pragma unroll
    for (int st = 0; st < kMaxSteps; ++st)
        if (ids[st] >= 0) atomicAdd(hist + ids[st], 1);
    __syncwarp();
    for (int e = lane; e < E; e += 32) ecount[static_cast<int64_t>(e) * chunks_pad + chunk] = hist[e];
}

__global__ void __launch_bounds__(kThreads)
expert_scan_kernel(int32_t P, int32_t E, int64_t chunks, int64_t chunks_pad, const int32_t* __restrict__ reo,
                   const int32_t* __restrict__ nrtpe, const int32_t* __restrict__ ecount,
                   int32_t* __restrict__ ebase, int64_t* __restrict__ expert_part_base) {
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw < E) {
        const int64_t e = gw;
        const int32_t* col = ecount + e * chunks_pad;
        int32_t carry = __ldg(reo + e);
        for (int64_t c0 = 0; c0 < chunks; c0 += 32 * kSeg) {
            const int64_t cb = c0 + static_cast<int64_t>(lane) * kSeg;
            int32_t v[kSeg];
#pragma unroll
            for (int q = 0; q < kSeg; q += 4) {
                // cb + q is a multiple of 4 and so is the row stride: whole int4 inside the row
                const int4 u = cb + q < chunks_pad ? __ldg(reinterpret_cast<const int4*>(col + cb + q))
                                                   : make_int4(0, 0, 0, 0);
                v[q] = u.x;
                v[q + 1] = u.y;
                v[q + 2] = u.z;
                v[q + 3] = u.w;
            }
            int32_t sum = 0;
#pragma unroll
            for (int u = 0; u < kSeg; ++u) {
                if (cb + u >= chunks) v[u] = 0;  // row padding
                sum += v[u];
            }
            int32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            int32_t run = carry + incl - sum;
#pragma unroll
            for (int u = 0; u < kSeg; ++u) {
                if (cb + u < chunks) ebase[(cb + u) * E + e] = run;
                run += v[u];
            }
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
    const int64_t g0 = chunk * kChunkTokens;
    const int64_t g1 = g0 + kChunkTokens < S ? g0 + kChunkTokens : S;
    const int nslots = static_cast<int>((g1 - g0) * K);
    int32_t ids[kMaxSteps];
    load_chunk(topk_idx, g0 * K, nslots, E, lane, ids);
    for (int e = lane; e < E; e += 32) next[e] = __ldg(ebase + chunk * E + e);
    __syncwarp();
    const uint32_t below = lanemask_lt();
    int32_t* out = slot_row + g0 * K;
#pragma unroll
    for (int st = 0; st < kMaxSteps; ++st) {
        if (st * 32 >= nslots) break;  // warp-uniform
        const int f = st * 32 + lane;
        const int32_t e = ids[st];
        const uint32_t grp = __match_any_sync(0xffffffffu, e);
        if (f < nslots) out[f] = e >= 0 ? next[e] + __popc(grp & below) : -1;
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(grp)) next[e] += __popc(grp);
        __syncwarp();
    }
}

}  // namespace

int64_t notify_expert_scratch_bytes(const moe_shape& s) { return expert_plan(s).scratch_bytes; }

cudaError_t launch_notify_expert(const moe_shape& s, const int32_t* topk_idx, const int32_t* nrtpe,
                                 const int32_t* reo, int32_t* slot_row, int64_t* expert_part_base,
                                 void* scratch, cudaStream_t stream) {
    const ExpertPlan p = expert_plan(s);
    int32_t* ecount = static_cast<int32_t*>(scratch);
    int32_t* ebase = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) + p.ebase_off);
    cudaError_t e = cudaSuccess;
    if (p.chunks > 0) {
        e = prepare_kernel(reinterpret_cast<const void*>(expert_count_kernel), p.smem, p.wpb * 32, nullptr);
        if (e != cudaSuccess) return e;
        e = prepare_kernel(reinterpret_cast<const void*>(expert_rows_kernel), p.smem, p.wpb * 32, nullptr);
        if (e != cudaSuccess) return e;
        e = launch_pdl(expert_count_kernel, static_cast<unsigned>(p.blocks), p.wpb * 32, p.smem, stream, s.E,
                       s.K, static_cast<int64_t>(s.S), p.chunks, p.chunks_pad, topk_idx, ecount);
        if (e != cudaSuccess) return e;
    }
    const int64_t scan_warps = static_cast<int64_t>(s.E) + 1;
    e = launch_pdl(expert_scan_kernel, static_cast<unsigned>(ceil_div(scan_warps, kThreads / 32)), kThreads, 0,
                   stream, s.P, s.E, p.chunks, p.chunks_pad, reo, nrtpe, static_cast<const int32_t*>(ecount), ebase,
                   expert_part_base);
    if (e != cudaSuccess || p.chunks == 0) return e;
    return launch_pdl(expert_rows_kernel, static_cast<unsigned>(p.blocks), p.wpb * 32, p.smem, stream, s.E, s.K,
                      static_cast<int64_t>(s.S), p.chunks, topk_idx, static_cast<const int32_t*>(ebase), slot_row);
}

MOE_PROFILE_UNIT(expert)

}  // namespace moe
