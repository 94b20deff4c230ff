// layout.cu -- routing tables from topk_idx (moe_layout).
//
// Computes, per source rank s, num_tokens_per_rank[s][d], num_tokens_per_expert[s][e]
// and the token -> rank table is_token_in_rank[g][d] (plus its packed form), as
// described in "Ascend DeepEP MoE Dispatch Optimization", sections
// "从 Python 接口进入真实调用链" and "Dispatch handle 六项分别保存什么"; the
// destination rank of an expert is expert_id / experts_per_rank (section
// "一条 token 如何走完 MoE").
//
// Design (sm_103a): one thread per token, blocks never straddle source ranks.
//  * Expert histogram: one shared-memory histogram per block, each (token, k)
//    slot adds 1 with an integer atomic (the counts do not depend on the order).
//  * Rank counts: one __ballot_sync + __popc per rank over the warp's tokens,
//    summed over the block's warps in a fixed order.
//  * Block partials go to scratch and a second kernel sums them in block
//    order: the result is the same on every run.
//  * The block's slice of is_token_in_rank (and of the packed bits) is built in
//    shared memory and written out with 16-byte stores: the slice of rows
//    [g0, g0+n) is one contiguous span.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kLayoutMaxThreads = 256;
constexpr int kReduceThreads = 256;

struct LayoutSmem {
    size_t off_bits, off_itr, total;
};

__host__ __device__ inline LayoutSmem layout_smem(int P, int E, int tb) {
    const int nwarps = tb / 32;
    const int W = (P + 31) / 32;
    LayoutSmem l;
    l.off_bits = static_cast<size_t>(round_up((static_cast<int64_t>(nwarps) * P + E) * 4, 16));
    l.off_itr = l.off_bits + static_cast<size_t>(tb) * W * 4;
    l.total = l.off_itr + static_cast<size_t>(round_up(static_cast<int64_t>(tb) * P, 16));
    return l;
}

__device__ inline void copy_bytes_out(uint8_t* dst, const uint8_t* src, int64_t nbytes, int tid,
                                      int nthreads) {
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        const int64_t nv = nbytes >> 4;
        for (int64_t i = tid; i < nv; i += nthreads)
            reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
        for (int64_t i = (nv << 4) + tid; i < nbytes; i += nthreads) dst[i] = src[i];
    } else {
        for (int64_t i = tid; i < nbytes; i += nthreads) dst[i] = src[i];
    }
}

__global__ void __launch_bounds__(kLayoutMaxThreads)
layout_count_kernel(int32_t P, int32_t E, int32_t K, int64_t T, int64_t nbs, int64_t part_stride,
                    const int32_t* __restrict__ topk_idx, uint8_t* __restrict__ itr,
                    uint32_t* __restrict__ bits, int32_t* __restrict__ part) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) unsigned char smem[];
    const int tb = blockDim.x;
    const int nwarps = tb >> 5;
    const int W = (P + 31) >> 5;
    const int epr = E / P;
    const LayoutSmem L = layout_smem(P, E, tb);
    int32_t* hist_rank = reinterpret_cast<int32_t*>(smem);   // [nwarps][P]
    int32_t* hist_exp = hist_rank + nwarps * P;               // [E], whole block
    uint32_t* tile_bits = reinterpret_cast<uint32_t*>(smem + L.off_bits);  // [tb][W]
    uint8_t* tile_itr = smem + L.off_itr;                                   // [tb][P]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t s = blockIdx.x / nbs;
    const int64_t t0 = (blockIdx.x % nbs) * tb;
    const int n = static_cast<int>(min(static_cast<int64_t>(tb), T - t0));
    const int64_t g0 = s * T + t0;

    for (size_t i = tid; i < L.total / 4; i += tb) reinterpret_cast<uint32_t*>(smem)[i] = 0u;
    __syncthreads();

    const bool active = tid < n;
    const int64_t g = g0 + tid;
    int bad = 0;
    uint8_t* my_row = tile_itr + tid * P;
    uint32_t* my_bits = tile_bits + tid * W;
    for (int k = 0; k < K; ++k) {
        const int32_t e = active ? __ldg(topk_idx + g * K + k) : -1;
        if (e >= E) bad = 1;
        if (e >= 0 && e < E) {
            atomicAdd(hist_exp + e, 1);
            const int d = e / epr;
            my_row[d] = 1;
            my_bits[d >> 5] |= 1u << (d & 31);
        }
    }
    __syncwarp();
    // Tokens of this warp per rank: one ballot per rank.
    for (int wd = 0; wd < W; ++wd) {
        const uint32_t word = my_bits[wd];
        const int dn = min(32, P - wd * 32);
        for (int j = 0; j < dn; ++j) {
            const uint32_t bal = __ballot_sync(0xffffffffu, (word >> j) & 1u);
            if (lane == j) hist_rank[warp * P + wd * 32 + j] = __popc(bal);
        }
    }
    const int any_bad = __syncthreads_or(bad);

    copy_bytes_out(itr + g0 * P, tile_itr, static_cast<int64_t>(n) * P, tid, tb);
    if (bits) {
        uint32_t* dst = bits + g0 * W;
        for (int i = tid; i < n * W; i += tb) dst[i] = tile_bits[i];
    }
    int32_t* mine = part + static_cast<int64_t>(blockIdx.x) * part_stride;
    for (int j = tid; j < P; j += tb) {
        int32_t sum = 0;
        for (int w = 0; w < nwarps; ++w) sum += hist_rank[w * P + j];
        mine[j] = sum;
    }
    for (int j = tid; j < E; j += tb) mine[P + j] = hist_exp[j];
    if (tid == 0) mine[P + E] = any_bad;
}

// Sum the block partials of each source rank in block order; block 0 also
// folds the blocks' error flags into the caller's error word.
__global__ void __launch_bounds__(kReduceThreads)
layout_reduce_kernel(int32_t P, int32_t E, int64_t nbs, int64_t part_stride,
                     const int32_t* __restrict__ part, int32_t* __restrict__ ntpr,
                     int32_t* __restrict__ ntpe, int32_t* __restrict__ err) {
    pdl_wait_then_release();
    const int64_t s = blockIdx.x;
    const int32_t* base = part + s * nbs * part_stride;
    for (int j = threadIdx.x; j < P + E; j += blockDim.x) {
        int32_t sum = 0;
#pragma unroll 8
        for (int64_t b = 0; b < nbs; ++b) sum += base[b * part_stride + j];
        if (j < P)
            ntpr[s * P + j] = sum;
        else
            ntpe[s * E + (j - P)] = sum;
    }
    if (blockIdx.x == 0) {
        int bad = 0;
        const int64_t nblk = static_cast<int64_t>(P) * nbs;
        for (int64_t i = threadIdx.x; i < nblk; i += blockDim.x) bad |= part[i * part_stride + P + E];
        bad = __syncthreads_or(bad);
        if (threadIdx.x == 0 && err) *err = bad ? MOE_ERR_TOPK_OUT_OF_RANGE : MOE_OK;
    }
}

}  // namespace

LayoutPlan layout_plan(const moe_shape& s) {
    LayoutPlan p;
    const int64_t T = s.S / s.P;
    int tb = (32768 / s.P) / 32 * 32;
    tb = tb < 32 ? 32 : (tb > kLayoutMaxThreads ? kLayoutMaxThreads : tb);
    p.threads = tb;
    p.blocks_per_source = T > 0 ? ceil_div(T, tb) : 0;
    p.part_stride = static_cast<int64_t>(s.P) + s.E + 1;
    p.smem = layout_smem(s.P, s.E, tb).total;
    p.scratch_bytes = round_up(static_cast<int64_t>(s.P) * p.blocks_per_source * p.part_stride * 4, 256);
    return p;
}

cudaError_t launch_layout(const moe_shape& s, const int32_t* topk_idx, int32_t* ntpr, int32_t* ntpe,
                          uint8_t* itr, uint32_t* bits, int32_t* err, void* scratch,
                          cudaStream_t stream) {
    const LayoutPlan p = layout_plan(s);
    int32_t* part = static_cast<int32_t*>(scratch);
    const int64_t blocks = static_cast<int64_t>(s.P) * p.blocks_per_source;
    cudaError_t e = cudaSuccess;
    if (blocks > 0) {
        e = prepare_kernel(reinterpret_cast<const void*>(layout_count_kernel), p.smem, p.threads, nullptr);
        if (e != cudaSuccess) return e;
        e = launch_pdl(layout_count_kernel, static_cast<unsigned>(blocks), p.threads, p.smem, stream, s.P,
                       s.E, s.K, static_cast<int64_t>(s.S / s.P), p.blocks_per_source, p.part_stride,
                       topk_idx, itr, bits, part);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(layout_reduce_kernel, static_cast<unsigned>(s.P), kReduceThreads, 0, stream, s.P, s.E,
                      p.blocks_per_source, p.part_stride, static_cast<const int32_t*>(part), ntpr, ntpe, err);
}

}  // namespace moe
