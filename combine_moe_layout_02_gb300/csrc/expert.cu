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
// Two launches over chunks of up to kChunk consecutive tokens (the plan's
// power of two giving about 64 chunks), one CTA per chunk and one thread per
// token (a token's K slots are contiguous in topk_idx):
//  1. count: the chunk's expert histogram (shared-memory integer atomics)
//     into scratch, expert-major: ecount[e][chunk];
//  2. rows: each CTA adds, per expert, the counts of the chunks before its own
//     (its row of ecount, 16-byte loads) to recv_expert_offset -- the chunk's
//     first row of every expert; per-warp histograms of the chunk become
//     exclusive warp offsets; then each warp ranks its slots 32 at a time in
//     (token, k) order among the step's slots of the same expert: each lane
//     sets its bit in the warp's shared-memory mask of its expert, reads the
//     mask back (the lanes of its group) and takes the popcount of the lower
//     lanes; the group's last lane advances the expert's offset and clears the
//     mask. (__match_any_sync gives the same groups; measured on GB300 it cost
//     about 1000 cycles a step.) CTA 0 also scans the rank totals into
//     expert_part_base.
// Integer counts: the result does not depend on the order of the atomics.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kChunk = 1024;   // tokens per chunk = threads per CTA
constexpr int kWarps = kChunk / 32;

struct ExpertPlan {
    int64_t chunks, chunks_pad;  // chunk count; expert-major row stride (a multiple of 4)
    int threads;                 // kChunk, or fewer (a multiple of 32) when S is smaller
    size_t smem_count, smem_rows;
    int64_t scratch_bytes;
};

ExpertPlan expert_plan(const moe_shape& s) {
    ExpertPlan p;
    // One token per thread and about 64 chunks (measured best at S = 4096,
    // 32768 and 65536: fewer chunks leave SMs idle, more lengthen each CTA's
    // prefix over the earlier chunks): a power of two from 256 to kChunk, no
    // more than S needs, and few enough warps that their histograms and group
    // masks (2 x [warps][E]) stay within 128 KB.
    int64_t t = 256;
    while (t < kChunk && t * 64 < s.S) t <<= 1;
    if (t > s.S) t = round_up(s.S > 0 ? s.S : 1, 32);
    const int64_t by_smem = (128 * 1024 / (static_cast<int64_t>(s.E) * 8)) * 32;
    if (t > by_smem) t = by_smem < 32 ? 32 : by_smem / 32 * 32;
    p.threads = static_cast<int>(t);
    p.chunks = ceil_div(s.S, t);
    p.chunks_pad = round_up(p.chunks, 4);
    p.smem_count = static_cast<size_t>(s.E) * 4;
    // per-warp histograms [warps][E], the chunk's bases [E], slot ids
    // [threads][K] and per-warp group masks [warps][E]
    p.smem_rows = (static_cast<size_t>(p.threads / 32) + 1) * s.E * 4 + static_cast<size_t>(p.threads) * s.K * 4 +
                  static_cast<size_t>(p.threads / 32) * s.E * 4;
    p.scratch_bytes = round_up(static_cast<int64_t>(s.E) * p.chunks_pad * 4, 256);
    return p;
}

// Token g's K expert ids (out-of-range and masked ids as -1), 16-byte loads
// when K is a multiple of 4.
__device__ __forceinline__ void load_ids(const int32_t* __restrict__ topk_idx, int64_t g, bool active, int K, int E,
                                         int32_t (&ids)[MOE_MAX_TOPK]) {
    if ((K & 3) == 0) {
#pragma unroll
        for (int k4 = 0; k4 < MOE_MAX_TOPK; k4 += 4) {
            if (k4 < K) {
                const int4 v = active ? __ldg(reinterpret_cast<const int4*>(topk_idx + g * K + k4))
                                      : make_int4(-1, -1, -1, -1);
                ids[k4] = v.x;
                ids[k4 + 1] = v.y;
                ids[k4 + 2] = v.z;
                ids[k4 + 3] = v.w;
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < MOE_MAX_TOPK; ++k)
            if (k < K) ids[k] = active ? __ldg(topk_idx + g * K + k) : -1;
    }
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k)
        if (k < K && (ids[k] < 0 || ids[k] >= E)) ids[k] = -1;
}

__global__ void __launch_bounds__(kChunk)
expert_count_kernel(int32_t E, int32_t K, int64_t S, int64_t chunks_pad, const int32_t* __restrict__ topk_idx,
                    int32_t* __restrict__ ecount) {
    pdl_wait_then_release();
    MOE_PROF_BEGIN(kProfExpertCount);
    extern __shared__ __align__(16) int32_t hist[];  // [E]
    const int tid = threadIdx.x;
    const int64_t chunk = blockIdx.x;
    const int64_t g = chunk * blockDim.x + tid;
    int32_t ids[MOE_MAX_TOPK];
    load_ids(topk_idx, g, g < S, K, E, ids);
    for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k)
        if (k < K && ids[k] >= 0) atomicAdd(hist + ids[k], 1);
    MOE_STAMP(1);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) ecount[static_cast<int64_t>(e) * chunks_pad + chunk] = hist[e];
    MOE_STAMP(2);
    MOE_PROF_END_N(3);
}

__global__ void __launch_bounds__(kChunk)
expert_rows_kernel(int32_t P, int32_t E, int32_t K, int64_t S, int64_t chunks, int64_t chunks_pad,
                   const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ ecount,
                   const int32_t* __restrict__ reo, const int32_t* __restrict__ nrtpe, int32_t* __restrict__ slot_row,
                   int64_t* __restrict__ expert_part_base) {
    pdl_wait_then_release();
    MOE_PROF_BEGIN(kProfNotifyExpert);
    extern __shared__ __align__(16) int32_t sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    int32_t* whist = sm;                       // [nwarps][E]: counts, then each warp's first rows
    int32_t* cbase = sm + nwarps * E;          // [E]: the chunk's first row of each expert
    int32_t* sids = cbase + E;                 // [threads][K]: the chunk's slot ids in (token, k) order
    uint32_t* gmask = reinterpret_cast<uint32_t*>(sids + blockDim.x * K);  // [nwarps][E]: lanes per expert
    const int64_t chunk = blockIdx.x;
    const int64_t g0 = chunk * blockDim.x;
    const bool work = chunk < chunks;

    if (chunk == 0) {  // the expert-major partition bases, from the aligned counts
        if (warp == nwarps - 1) {
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
    if (!work) {
        MOE_PROF_END_N(1);
        return;
    }

    const int64_t g = g0 + tid;
    int32_t ids[MOE_MAX_TOPK];
    load_ids(topk_idx, g, g < S, K, E, ids);
    // Chunk base of each expert: its first receive row plus the slots of the
    // earlier chunks (this CTA's prefix of the expert's ecount row).
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t acc = __ldg(reo + e);
        const int32_t* row = ecount + static_cast<int64_t>(e) * chunks_pad;
        int64_t c = 0;
#pragma unroll 16
        for (; c + 4 <= chunk; c += 4) {
            const int4 v = __ldg(reinterpret_cast<const int4*>(row + c));
            acc += v.x + v.y + v.z + v.w;
        }
        for (; c < chunk; ++c) acc += __ldg(row + c);
        cbase[e] = acc;
    }
    MOE_STAMP(1);
    for (int i = tid; i < nwarps * E; i += blockDim.x) {
        whist[i] = 0;
        gmask[i] = 0u;
    }
    int32_t* srow = sids + tid * K;
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k)
        if (k < K) srow[k] = ids[k];
    __syncthreads();
    int32_t* my = whist + warp * E;
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k)
        if (k < K && ids[k] >= 0) atomicAdd(my + ids[k], 1);
    __syncthreads();
    MOE_STAMP(2);
    // Exclusive warp offsets per expert, from the chunk base.
    for (int e = tid; e < E; e += blockDim.x) {
        int32_t run = cbase[e];
        for (int w = 0; w < nwarps; ++w) {
            const int32_t v = whist[w * E + e];
            whist[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    MOE_STAMP(3);
    // Rank each slot among the earlier slots of its expert, 32 slots a step.
    const int64_t wg0 = g0 + warp * 32;  // the warp's first token
    const int ntok = static_cast<int>(min(static_cast<int64_t>(32), S - wg0));
    if (ntok <= 0) {
        MOE_STAMP(4);
        MOE_PROF_END_N(5);
        return;
    }
    const int nslots = ntok * K;
    const int32_t* wids = sids + warp * 32 * K;
    int32_t* out = slot_row + wg0 * K;
    const uint32_t below = lanemask_lt();
    uint32_t* wm = gmask + warp * E;
    for (int f0 = 0; f0 < nslots; f0 += 32) {
        const int f = f0 + lane;
        const int32_t e = f < nslots ? wids[f] : -1;
        if (e >= 0) atomicOr(wm + e, 1u << lane);
        __syncwarp();
        const uint32_t grp = e >= 0 ? wm[e] : 0u;  // the lanes of this step with expert e
        if (f < nslots) out[f] = e >= 0 ? my[e] + __popc(grp & below) : -1;
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(grp)) {
            my[e] += __popc(grp);
            wm[e] = 0u;
        }
        __syncwarp();
    }
    MOE_STAMP(4);
    MOE_PROF_END_N(5);
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
        e = prepare_kernel(reinterpret_cast<const void*>(expert_count_kernel), p.smem_count, p.threads, nullptr);
        if (e != cudaSuccess) return e;
        e = launch_pdl(expert_count_kernel, static_cast<unsigned>(p.chunks), p.threads, p.smem_count, stream, s.E,
                       s.K, static_cast<int64_t>(s.S), p.chunks_pad, topk_idx, ecount);
        if (e != cudaSuccess) return e;
    }
    e = prepare_kernel(reinterpret_cast<const void*>(expert_rows_kernel), p.smem_rows, p.threads, nullptr);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.chunks > 0 ? p.chunks : 1);
    return launch_pdl(expert_rows_kernel, grid, p.threads, p.smem_rows, stream, s.P, s.E, s.K,
                      static_cast<int64_t>(s.S), p.chunks, p.chunks_pad, topk_idx,
                      static_cast<const int32_t*>(ecount), reo, nrtpe, slot_row, expert_part_base);
}

MOE_PROFILE_UNIT(expert)

}  // namespace moe
