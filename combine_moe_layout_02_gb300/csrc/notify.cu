// notify.cu -- counts and prefixes (moe_notify).
//
// "Ascend DeepEP MoE Dispatch Optimization", section "Notify 先交换数量和前缀":
// notify turns the routing into how many rows each rank receives, how many per
// local expert, and where each (source rank, channel) segment starts. Section
// "Device 侧如何把 channel 变成远端 Put" gives the receive position of a row:
// rank_prefix_matrix[s-1][d] + channel_prefix_matrix[s][d][c-1] + the running
// count inside channel c. "internode.cu", section 1 (notify_dispatch) rounds
// the per-expert receive counts up to expert_alignment. Channel c of a source
// rank is the c-th block of the balanced split of "HCCL Window 模式
// (Non-SHMEM) 代码深度剖析", section 8.3.
//
// Two launches, both one block per (source rank, channel):
//  1. notify_count_kernel: per-rank counts of the channel's tokens (warp
//     ballots into per-warp shared counters, fixed-order block sum) into
//     scratch. One extra block computes the rank prefix matrix, receive
//     totals, packed partition bases and the per-expert counts and offsets.
//  2. notify_head_kernel: channel prefixes from the scratch counts, then
//     send_head for the channel's tokens: ballot + popc of the lanes below
//     (rank inside the warp), an exclusive scan over the block's warps and a
//     running carry across block-sized chunks.
// No atomics: every output is a fixed-order integer sum.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kNotifyThreads = 256;
constexpr int kNotifyWarps = kNotifyThreads / 32;

// For each rank d, ballot "token of this lane is bound for d" over the warp and
// hand the ballot to f(d, ballot). Loads the token's row 4 bytes at a time
// when P is a multiple of 4 (rows then start 4-byte aligned).
template <typename F>
__device__ __forceinline__ void for_each_rank_ballot(const uint8_t* row, bool active, int P, F&& f) {
    if ((P & 3) == 0) {
        for (int d4 = 0; d4 < P; d4 += 4) {
            const uint32_t w4 = active ? __ldg(reinterpret_cast<const uint32_t*>(row + d4)) : 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t bal = __ballot_sync(0xffffffffu, ((w4 >> (8 * j)) & 0xffu) != 0u);
                f(d4 + j, bal);
            }
        }
    } else {
        for (int d = 0; d < P; ++d) {
            const uint32_t bal = __ballot_sync(0xffffffffu, active && __ldg(row + d) != 0);
            f(d, bal);
        }
    }
}

// The extra block of notify_count_kernel: everything that only depends on the
// per-source count matrices.
__device__ void notify_prefix_block(int32_t P, int32_t E, int32_t A, const int32_t* __restrict__ ntpr,
                                    const int32_t* __restrict__ ntpe, int32_t* __restrict__ rpm,
                                    int32_t* __restrict__ nrt, int32_t* __restrict__ nrtpe,
                                    int32_t* __restrict__ reo, int64_t* __restrict__ part_row_base,
                                    int32_t* tot /* shared, [P] */) {
    __shared__ int64_t warp_sum[kNotifyWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int epr = E / P;
    for (int d = tid; d < P; d += nthreads) {
        int32_t run = 0;
#pragma unroll 8
        for (int s = 0; s < P; ++s) {
            run += ntpr[s * P + d];
            rpm[s * P + d] = run;
        }
        nrt[d] = run;
        tot[d] = run;
    }
    for (int e = tid; e < E; e += nthreads) {
        int64_t cnt = 0;
#pragma unroll 8
        for (int s = 0; s < P; ++s) cnt += ntpe[static_cast<int64_t>(s) * E + e];
        nrtpe[e] = static_cast<int32_t>(round_up(cnt, A));
    }
    __syncthreads();
    // Packed partition bases: exclusive scan of the receive totals.
    const int per = static_cast<int>(ceil_div(P, nthreads));
    const int d0 = min(P, tid * per), d1 = min(P, d0 + per);
    int64_t local = 0;
    for (int d = d0; d < d1; ++d) local += tot[d];
    int64_t incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int64_t before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    int64_t run = before + incl - local;
    for (int d = d0; d < d1; ++d) {
        part_row_base[d] = run;
        run += tot[d];
    }
    if (d0 < d1 && d1 == P) part_row_base[P] = run;
    // Per-expert offsets inside each rank.
    for (int d = tid; d < P; d += nthreads) {
        int32_t off = 0;
        for (int l = 0; l < epr; ++l) {
            reo[d * epr + l] = off;
            off += nrtpe[d * epr + l];
        }
    }
}

__global__ void __launch_bounds__(kNotifyThreads)
notify_count_kernel(int32_t P, int32_t E, int32_t C, int32_t A, int64_t T,
                    const int32_t* __restrict__ ntpr, const int32_t* __restrict__ ntpe,
                    const uint8_t* __restrict__ itr, int32_t* __restrict__ rpm,
                    int32_t* __restrict__ nrt, int32_t* __restrict__ nrtpe, int32_t* __restrict__ reo,
                    int64_t* __restrict__ part_row_base, int32_t* __restrict__ ccount) {
    extern __shared__ __align__(16) int32_t wcnt[];  // [warps][P]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    if (blockIdx.x == static_cast<unsigned>(P) * C) {
        notify_prefix_block(P, E, A, ntpr, ntpe, rpm, nrt, nrtpe, reo, part_row_base, wcnt);
        return;
    }
    const int64_t s = blockIdx.x / C, c = blockIdx.x % C;
    int64_t b, e;
    split_range(T, C, c, &b, &e);
    for (int i = tid; i < nwarps * P; i += nthreads) wcnt[i] = 0;
    __syncthreads();
    int32_t* mine = wcnt + warp * P;
    for (int64_t t0 = b; t0 < e; t0 += nthreads) {
        const int64_t t = t0 + tid;
        const bool active = t < e;
        const uint8_t* row = itr + (s * T + (active ? t : b)) * P;
        for_each_rank_ballot(row, active, P, [&](int d, uint32_t bal) {
            if (lane == (d & 31)) mine[d] += __popc(bal);
        });
    }
    __syncthreads();
    for (int d = tid; d < P; d += nthreads) {
        int32_t sum = 0;
        for (int w = 0; w < nwarps; ++w) sum += wcnt[w * P + d];
        ccount[static_cast<int64_t>(blockIdx.x) * P + d] = sum;
    }
}

__global__ void __launch_bounds__(kNotifyThreads)
notify_head_kernel(int32_t P, int32_t C, int64_t T, const uint8_t* __restrict__ itr,
                   const int32_t* __restrict__ rpm, const int32_t* __restrict__ ccount,
                   int32_t* __restrict__ cpm, int32_t* __restrict__ rcpm,
                   int32_t* __restrict__ send_head) {
    extern __shared__ __align__(16) int32_t sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    int32_t* base = sm;           // [P]   next free row of d for this channel
    int32_t* woff = sm + P;       // [warps][P]
    const int64_t s = blockIdx.x / C, c = blockIdx.x % C;
    int64_t b, e;
    split_range(T, C, c, &b, &e);
    for (int d = tid; d < P; d += nthreads) {
        int32_t pre = 0;
#pragma unroll 8
        for (int64_t cc = 0; cc < c; ++cc) pre += ccount[(s * C + cc) * P + d];
        const int32_t cnt = ccount[(s * C + c) * P + d];
        cpm[(s * P + d) * C + c] = pre + cnt;
        const int32_t rank_base = s > 0 ? rpm[(s - 1) * P + d] : 0;
        rcpm[(static_cast<int64_t>(d) * P + s) * C + c] = rank_base + pre;
        base[d] = rank_base + pre;
    }
    __syncthreads();
    int32_t* mine = woff + warp * P;
    for (int64_t t0 = b; t0 < e; t0 += nthreads) {
        const int64_t t = t0 + tid;
        const bool active = t < e;
        const int64_t g = s * T + (active ? t : b);
        const uint8_t* row = itr + g * P;
        for_each_rank_ballot(row, active, P, [&](int d, uint32_t bal) {
            if (lane == (d & 31)) mine[d] = __popc(bal);
        });
        __syncthreads();
        for (int d = tid; d < P; d += nthreads) {
            int32_t run = base[d];
            for (int w = 0; w < nwarps; ++w) {
                const int32_t cnt = woff[w * P + d];
                woff[w * P + d] = run;
                run += cnt;
            }
            base[d] = run;
        }
        __syncthreads();
        const uint32_t below = lanemask_lt();
        int32_t* out = send_head + g * P;
        if ((P & 3) == 0) {
            int4 pack;
            for_each_rank_ballot(row, active, P, [&](int d, uint32_t bal) {
                const bool has = (bal >> lane) & 1u;
                const int32_t v = has ? mine[d] + __popc(bal & below) : -1;
                switch (d & 3) {
                    case 0: pack.x = v; break;
                    case 1: pack.y = v; break;
                    case 2: pack.z = v; break;
                    default:
                        pack.w = v;
                        if (active) *reinterpret_cast<int4*>(out + (d - 3)) = pack;
                }
            });
        } else {
            for_each_rank_ballot(row, active, P, [&](int d, uint32_t bal) {
                const bool has = (bal >> lane) & 1u;
                if (active) out[d] = has ? mine[d] + __popc(bal & below) : -1;
            });
        }
        __syncthreads();
    }
}

}  // namespace

int64_t notify_scratch_bytes(const moe_shape& s) {
    return round_up(static_cast<int64_t>(s.P) * s.num_channels * s.P * 4, 256);
}

cudaError_t launch_notify(const moe_shape& s, const int32_t* ntpr, const int32_t* ntpe,
                          const uint8_t* itr, int32_t* rpm, int32_t* cpm, int32_t* rcpm,
                          int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                          int64_t* part_row_base, void* scratch, cudaStream_t stream) {
    const int64_t T = s.S / s.P;
    int32_t* ccount = static_cast<int32_t*>(scratch);
    const int64_t chans = static_cast<int64_t>(s.P) * s.num_channels;
    const size_t smem_count = static_cast<size_t>(kNotifyWarps) * s.P * 4;
    const size_t smem_head = static_cast<size_t>(kNotifyWarps + 1) * s.P * 4;
    cudaError_t e = cudaFuncSetAttribute(notify_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_count));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(notify_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_head));
    if (e != cudaSuccess) return e;
    notify_count_kernel<<<static_cast<unsigned>(chans + 1), kNotifyThreads, smem_count, stream>>>(
        s.P, s.E, s.num_channels, s.expert_alignment, T, ntpr, ntpe, itr, rpm, nrt, nrtpe, reo,
        part_row_base, ccount);
    notify_head_kernel<<<static_cast<unsigned>(chans), kNotifyThreads, smem_head, stream>>>(
        s.P, s.num_channels, T, itr, rpm, ccount, cpm, rcpm, send_head);
    return cudaGetLastError();
}

}  // namespace moe
