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
// Two launches. Work is handed out per warp, so every block shape works:
//  1. notify_count_kernel
//     - channel part: per-rank token counts of each (source rank, channel)
//       into scratch;
//     - rank part: one warp per destination column scans num_tokens_per_rank
//       down the source ranks (warp-shuffle scan with a carry) into
//       rank_prefix_matrix and num_recv_tokens;
//     - expert part: one warp per expert sums num_tokens_per_expert over
//       source ranks and rounds up to expert_alignment.
//  2. notify_head_kernel
//     - channel part: channel prefixes from the scratch counts, then
//       send_head for the channel's tokens;
//     - tail part: one warp per rank scans its per-expert counts into
//       recv_expert_offset; warp 0 scans the receive totals into the packed
//       partition bases.
// The channel part has two shapes:
//   * token-major (P < 32 or P % 4 != 0): one block per channel, one thread
//     per token; per rank a __ballot_sync, __popc of the lower lanes for the
//     rank inside the warp, and a scan over the block's warps;
//   * rank-major (P >= 32, P % 4 == 0): one warp per channel, each lane owns 4
//     ranks and walks the channel's tokens in order with 4 running counters;
//     a token's send_head row is one coalesced 16-byte store per lane.
// No atomics: every output is a fixed-order integer sum.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kMaxThreads = 256;

struct NotifyPlan {
    bool rank_major;
    int threads;             // block size
    int wpb;                 // warps per block
    int64_t chan_blocks;     // blocks of the channel part
    int64_t rank_blocks;     // kernel 1: rank-prefix blocks
    int64_t expert_blocks;   // kernel 1: expert-sum blocks
    int64_t tail_blocks;     // kernel 2: offset / base blocks
};

NotifyPlan notify_plan(const moe_shape& s) {
    NotifyPlan p;
    const int64_t T = s.S / s.P;
    const int64_t chans = static_cast<int64_t>(s.P) * s.num_channels;
    p.rank_major = s.P >= 32 && (s.P % 4) == 0;
    if (p.rank_major) {
        p.threads = kMaxThreads;
    } else {
        int64_t t = round_up(ceil_div(T, s.num_channels), 32);
        p.threads = static_cast<int>(t < 32 ? 32 : (t > kMaxThreads ? kMaxThreads : t));
    }
    p.wpb = p.threads / 32;
    p.chan_blocks = p.rank_major ? ceil_div(chans, p.wpb) : chans;
    p.rank_blocks = ceil_div(s.P, p.wpb);
    p.expert_blocks = ceil_div(s.E, p.wpb);
    p.tail_blocks = ceil_div(s.P, p.wpb);
    return p;
}

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

template <typename V>
__device__ __forceinline__ V warp_inclusive_scan(V v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__device__ __forceinline__ int flag(uint32_t w, int j) { return ((w >> (8 * j)) & 0xffu) != 0u; }

// ---- kernel 1 -------------------------------------------------------------

__global__ void __launch_bounds__(kMaxThreads)
notify_count_kernel(int32_t P, int32_t E, int32_t C, int32_t A, int64_t T, bool rank_major,
                    int64_t chan_blocks, int64_t rank_blocks, const int32_t* __restrict__ ntpr,
                    const int32_t* __restrict__ ntpe, const uint8_t* __restrict__ itr,
                    int32_t* __restrict__ rpm, int32_t* __restrict__ nrt, int32_t* __restrict__ nrtpe,
                    int32_t* __restrict__ ccount) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) int32_t wcnt[];  // token-major: [warps][P]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int wpb = nthreads >> 5;
    const int64_t bid = blockIdx.x;

    if (bid >= chan_blocks) {
        if (bid < chan_blocks + rank_blocks) {
            // Rank part: column d of num_tokens_per_rank, scanned over sources.
            const int64_t gw = (bid - chan_blocks) * wpb + warp;
            if (gw >= P) return;
            const int d = static_cast<int>(gw);
            int32_t carry = 0;
            for (int s0 = 0; s0 < P; s0 += 32) {
                const int s = s0 + lane;
                const int32_t v = s < P ? __ldg(ntpr + static_cast<int64_t>(s) * P + d) : 0;
                const int32_t incl = warp_inclusive_scan(v, lane);
                if (s < P) rpm[static_cast<int64_t>(s) * P + d] = carry + incl;
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) nrt[d] = carry;
        } else {
            // Expert part: receive count of expert e, summed over sources, aligned.
            const int64_t gw = (bid - chan_blocks - rank_blocks) * wpb + warp;
            if (gw >= E) return;
            int64_t sum = 0;
            for (int s = lane; s < P; s += 32) sum += __ldg(ntpe + static_cast<int64_t>(s) * E + gw);
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) nrtpe[gw] = static_cast<int32_t>(round_up(sum, A));
        }
        return;
    }

    if (rank_major) {
        const int64_t ch = bid * wpb + warp;
        if (ch >= static_cast<int64_t>(P) * C) return;
        const int64_t s = ch / C, c = ch % C;
        int64_t b, e;
        split_range(T, C, c, &b, &e);
        for (int d0 = 0; d0 < P; d0 += 128) {
            const int d = d0 + 4 * lane;
            if (d >= P) continue;
            int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll 8
            for (int64_t t = b; t < e; ++t) {
                const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(itr + (s * T + t) * P + d));
                c0 += flag(w, 0);
                c1 += flag(w, 1);
                c2 += flag(w, 2);
                c3 += flag(w, 3);
            }
            *reinterpret_cast<int4*>(ccount + ch * P + d) = make_int4(c0, c1, c2, c3);
        }
        return;
    }

    // Token-major channel counts.
    const int64_t s = bid / C, c = bid % C;
    int64_t b, e;
    split_range(T, C, c, &b, &e);
    for (int i = tid; i < wpb * P; i += nthreads) wcnt[i] = 0;
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
        for (int w = 0; w < wpb; ++w) sum += wcnt[w * P + d];
        ccount[bid * P + d] = sum;
    }
}

// ---- kernel 2 -------------------------------------------------------------

__global__ void __launch_bounds__(kMaxThreads)
notify_head_kernel(int32_t P, int32_t E, int32_t C, int64_t T, bool rank_major, int64_t chan_blocks,
                   const uint8_t* __restrict__ itr, const int32_t* __restrict__ rpm,
                   const int32_t* __restrict__ nrt, const int32_t* __restrict__ nrtpe,
                   const int32_t* __restrict__ ccount, int32_t* __restrict__ cpm,
                   int32_t* __restrict__ rcpm, int32_t* __restrict__ send_head,
                   int32_t* __restrict__ reo, int64_t* __restrict__ part_row_base) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) int32_t sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthreads = blockDim.x;
    const int wpb = nthreads >> 5;
    const int64_t bid = blockIdx.x;

    if (bid >= chan_blocks) {
        // Tail part: per-rank expert offsets; warp 0 also the partition bases.
        const int64_t gw = (bid - chan_blocks) * wpb + warp;
        if (gw >= P) return;
        const int epr = E / P;
        const int64_t d = gw;
        int32_t carry = 0;
        for (int l0 = 0; l0 < epr; l0 += 32) {
            const int l = l0 + lane;
            const int32_t v = l < epr ? __ldg(nrtpe + d * epr + l) : 0;
            const int32_t incl = warp_inclusive_scan(v, lane);
            if (l < epr) reo[d * epr + l] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (gw == 0) {
            int64_t run = 0;
            for (int d0 = 0; d0 < P; d0 += 32) {
                const int dd = d0 + lane;
                const int64_t v = dd < P ? __ldg(nrt + dd) : 0;
                const int64_t incl = warp_inclusive_scan(v, lane);
                if (dd < P) part_row_base[dd] = run + incl - v;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) part_row_base[P] = run;
        }
        return;
    }

    if (rank_major) {
        const int64_t ch = bid * wpb + warp;
        if (ch >= static_cast<int64_t>(P) * C) return;
        const int64_t s = ch / C, c = ch % C;
        int64_t b, e;
        split_range(T, C, c, &b, &e);
        for (int d0 = 0; d0 < P; d0 += 128) {
            const int d = d0 + 4 * lane;
            if (d >= P) continue;
            int4 pre = make_int4(0, 0, 0, 0);
#pragma unroll 4
            for (int64_t cc = 0; cc < c; ++cc) {
                const int4 v = __ldg(reinterpret_cast<const int4*>(ccount + (s * C + cc) * P + d));
                pre.x += v.x;
                pre.y += v.y;
                pre.z += v.z;
                pre.w += v.w;
            }
            const int4 cnt = __ldg(reinterpret_cast<const int4*>(ccount + ch * P + d));
            const int4 rb = s > 0 ? __ldg(reinterpret_cast<const int4*>(rpm + (s - 1) * P + d))
                                  : make_int4(0, 0, 0, 0);
            cpm[(s * P + d + 0) * C + c] = pre.x + cnt.x;
            cpm[(s * P + d + 1) * C + c] = pre.y + cnt.y;
            cpm[(s * P + d + 2) * C + c] = pre.z + cnt.z;
            cpm[(s * P + d + 3) * C + c] = pre.w + cnt.w;
            int32_t b0 = rb.x + pre.x, b1 = rb.y + pre.y, b2 = rb.z + pre.z, b3 = rb.w + pre.w;
            rcpm[(static_cast<int64_t>(d + 0) * P + s) * C + c] = b0;
            rcpm[(static_cast<int64_t>(d + 1) * P + s) * C + c] = b1;
            rcpm[(static_cast<int64_t>(d + 2) * P + s) * C + c] = b2;
            rcpm[(static_cast<int64_t>(d + 3) * P + s) * C + c] = b3;
#pragma unroll 8
            for (int64_t t = b; t < e; ++t) {
                const int64_t g = s * T + t;
                const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(itr + g * P + d));
                int4 v;
                v.x = flag(w, 0) ? b0++ : -1;
                v.y = flag(w, 1) ? b1++ : -1;
                v.z = flag(w, 2) ? b2++ : -1;
                v.w = flag(w, 3) ? b3++ : -1;
                *reinterpret_cast<int4*>(send_head + g * P + d) = v;
            }
        }
        return;
    }

    // Token-major channel heads.
    int32_t* base = sm;      // [P]   next free row of d for this channel
    int32_t* woff = sm + P;  // [warps][P]
    const int64_t s = bid / C, c = bid % C;
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
            for (int w = 0; w < wpb; ++w) {
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
    const NotifyPlan p = notify_plan(s);
    int32_t* ccount = static_cast<int32_t*>(scratch);
    const size_t smem_count = p.rank_major ? 0 : static_cast<size_t>(p.wpb) * s.P * 4;
    const size_t smem_head = p.rank_major ? 0 : static_cast<size_t>(p.wpb + 1) * s.P * 4;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(notify_count_kernel), smem_count, p.threads,
                                   nullptr);
    if (e != cudaSuccess) return e;
    e = prepare_kernel(reinterpret_cast<const void*>(notify_head_kernel), smem_head, p.threads, nullptr);
    if (e != cudaSuccess) return e;
    const int64_t grid1 = p.chan_blocks + p.rank_blocks + p.expert_blocks;
    e = launch_pdl(notify_count_kernel, static_cast<unsigned>(grid1), p.threads, smem_count, stream, s.P,
                   s.E, s.num_channels, s.expert_alignment, T, p.rank_major, p.chan_blocks, p.rank_blocks,
                   ntpr, ntpe, itr, rpm, nrt, nrtpe, ccount);
    if (e != cudaSuccess) return e;
    const int64_t grid2 = p.chan_blocks + p.tail_blocks;
    return launch_pdl(notify_head_kernel, static_cast<unsigned>(grid2), p.threads, smem_head, stream, s.P, s.E,
                      s.num_channels, T, p.rank_major, p.chan_blocks, itr, static_cast<const int32_t*>(rpm),
                      static_cast<const int32_t*>(nrt), static_cast<const int32_t*>(nrtpe),
                      static_cast<const int32_t*>(ccount), cpm, rcpm, send_head, reo, part_row_base);
}

}  // namespace moe
