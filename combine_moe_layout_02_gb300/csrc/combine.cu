// combine.cu -- inverse permutation and weighted reduction (moe_combine).
//
//   out[g] = bf16_rne( sum over ranks d ascending with send_head[g][d] >= 0 of
//                      c[g][d] * f32(y[part_row_base[d] + send_head[g][d]]) )
//
// "HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 7.8 (ReadBufferAndWeightedSum):
// an FP32 accumulator, per returned row Cast -> Muls(weight) -> Add, one final
// CAST_RINT to BF16. With one copy per distinct rank ("Ascend DeepEP MoE
// Dispatch Optimization", section "一条 token 如何走完 MoE") a rank's weight is
// the binary32 sum, in ascending k, of the Top-K weights of the token's slots on
// that rank (1 when no weights are given). Products and sums are rounded
// separately (__fmul_rn / __fadd_rn), ranks are visited in ascending order,
// so the result is the same bit pattern on every run.
//
// Design (sm_103a): persistent grid, no block barriers. The unit of work is a
// token, or a (token, column half) when the tokens would take at least
// MOE_COMBINE_SPLIT_ROUNDS rounds of the launch's warps: a warp takes units u,
// u + warps, ..., and halves keep the last round nearly full (whole tokens
// left about half the warps idle for the last of ~14 rounds at 32768 tokens;
// with only a few rounds the second compaction per token costs more).
//  * The warp compacts the token's send_head row into (row address, weight)
//    pairs in ascending rank order (ballot, then the r-th set bit's lane hands
//    its pair to lane r), then broadcasts the pairs to every lane once.
//  * Each lane owns 16-byte column chunks: it issues the loads of kUnroll
//    chunks from all of the token's rows before reducing any of them, so up to
//    kUnroll x MAXR x 16 bytes per lane are in flight, and stores 16 bytes of
//    out per chunk.
//  * The routing words of the warp's next unit (send_head row, Top-K ids and
//    weights) are loaded before the current unit's rows, so their latency
//    overlaps the payload traffic.
#include <cuda_bf16.h>

#include "moe_device.cuh"

#ifndef MOE_COMBINE_THREADS
#define MOE_COMBINE_THREADS 256
#endif
#ifndef MOE_COMBINE_UNROLL
#define MOE_COMBINE_UNROLL 2
#endif
// Whole-token rounds per warp from which tokens are split into column halves.
#ifndef MOE_COMBINE_SPLIT_ROUNDS
#define MOE_COMBINE_SPLIT_ROUNDS 8
#endif

namespace moe {
namespace {

constexpr int kCombineThreads = MOE_COMBINE_THREADS;
constexpr int kUnroll = MOE_COMBINE_UNROLL;
constexpr int64_t kSplitRounds = MOE_COMBINE_SPLIT_ROUNDS;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Two binary32 values to two bf16 (round to nearest even), packed low/high.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

// One lane's routing words of a token: send_head of rank `lane` (the first 32
// ranks; further ranks are read during the compaction) and Top-K slot `lane`.
struct TokenRoute {
    int32_t sh0;  // rank layout: send_head of rank `lane`; expert layout: slot_row of slot `lane`
    int32_t idx;
    float w;
};

template <bool EXPERT>
__device__ __forceinline__ TokenRoute load_route(const CombineArgs& a, int64_t g, int lane) {
    TokenRoute r{-1, -1, 0.f};
    if (g < a.S) {
        if (EXPERT) {
            if (lane < a.K) r.sh0 = __ldg(a.slot_row + g * a.K + lane);
        } else {
            if (lane < a.P) r.sh0 = __ldg(a.send_head + g * a.P + lane);
        }
        if (lane < a.K) {
            r.idx = __ldg(a.topk_idx + g * a.K + lane);
            if (a.topk_weights) r.w = __ldg(a.topk_weights + g * a.K + lane);
        }
    }
    return r;
}

template <int MAXR, bool EXPERT>
__global__ void __launch_bounds__(kCombineThreads, MAXR >= 16 ? 1 : 2)
combine_kernel(const CombineArgs a, int split_shift) {
    pdl_wait_then_release();
    extern __shared__ __align__(16) int64_t prb[];  // [P+1]
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i <= a.P; i += blockDim.x) prb[i] = a.part_row_base[i];
    __syncthreads();
    const int nchunks = a.H / 8;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t units = a.S << split_shift;
    int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (tid >> 5);
    TokenRoute cur = load_route<EXPERT>(a, u >> split_shift, lane);
    for (; u < units; u += warps_total) {
        const int64_t g = u >> split_shift;
        const int part = static_cast<int>(u - (g << split_shift));
        const int cb = static_cast<int>((static_cast<int64_t>(nchunks) * part) >> split_shift);
        const int ce = static_cast<int>((static_cast<int64_t>(nchunks) * (part + 1)) >> split_shift);
        const TokenRoute nxt = load_route<EXPERT>(a, (u + warps_total) >> split_shift, lane);
        const int32_t dk = (cur.idx >= 0 && cur.idx < a.E) ? cur.idx / a.epr : -1;
        // Compaction: lane r ends up holding the r-th valid rank's row and weight.
        uint64_t my_row = 0;
        float my_coef = 0.f;
        int n = 0;
        // Candidates: ranks d = d0 + lane (rank layout) or slots k = lane
        // (expert layout, K <= 32: one pass).
        const int ncand = EXPERT ? a.K : a.P;
        for (int d0 = 0; d0 < ncand; d0 += 32) {
            const int d = d0 + lane;
            bool valid = false;
            int64_t row = 0;
            float c = 0.f;
            if (EXPERT) {
                const int32_t sr = cur.sh0;
                if (dk >= 0 && sr >= 0) {
                    const int64_t lo = prb[dk], hi = prb[dk + 1];
                    row = lo + sr;
                    valid = sr < hi - lo && row >= 0 && row < a.arena_rows;
                    if (!valid) raise_error(a.err, MOE_ERR_CAPACITY);
                }
                c = a.topk_weights ? cur.w : 1.f;
            } else {
                const int32_t sh = d0 == 0 ? cur.sh0 : (d < a.P ? __ldg(a.send_head + g * a.P + d) : -1);
                if (sh >= 0) {
                    const int64_t lo = prb[d], hi = prb[d + 1];
                    row = lo + sh;
                    valid = sh < hi - lo && row >= 0 && row < a.arena_rows;
                    if (!valid) raise_error(a.err, MOE_ERR_CAPACITY);
                }
                for (int k = 0; k < a.K; ++k) {
                    const int32_t dkk = __shfl_sync(0xffffffffu, dk, k);
                    const float wk = __shfl_sync(0xffffffffu, cur.w, k);
                    if (dkk == d) c = __fadd_rn(c, wk);
                }
                if (!a.topk_weights) c = 1.f;
            }
            const uint64_t rp = reinterpret_cast<uint64_t>(a.y + row * a.y_stride);
            const uint32_t bal = __ballot_sync(0xffffffffu, valid);
            const int cnt = __popc(bal);
            for (int r = 0; r < cnt; ++r) {
                const int src = __fns(bal, 0, r + 1);  // lane of the (r+1)-th valid rank
                const uint64_t p = __shfl_sync(0xffffffffu, rp, src);
                const float cc = __shfl_sync(0xffffffffu, c, src);
                if (lane == n + r) {
                    my_row = p;
                    my_coef = cc;
                }
            }
            n += cnt;
        }
        if (n > MAXR) {
            if (lane == 0) raise_error(a.err, MOE_ERR_INCONSISTENT);
            n = MAXR;
        }
        const uint8_t* rows[MAXR];
        float coef[MAXR];
#pragma unroll
        for (int r = 0; r < MAXR; ++r) {
            rows[r] = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, my_row, r));
            coef[r] = __shfl_sync(0xffffffffu, my_coef, r);
        }
        uint16_t* out = a.out + g * a.H;
        for (int j0 = cb + lane; j0 < ce; j0 += 32 * kUnroll) {
            uint4 v[kUnroll][MAXR];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int j = j0 + 32 * q;
#pragma unroll
                for (int r = 0; r < MAXR; ++r)
                    if (r < n && j < ce) v[q][r] = ld_stream_u4(rows[r] + static_cast<size_t>(j) * 16);
            }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int j = j0 + 32 * q;
                if (j < ce) {
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
                    for (int r = 0; r < MAXR; ++r) {
                        if (r < n) {
                            const uint32_t w4[4] = {v[q][r].x, v[q][r].y, v[q][r].z, v[q][r].w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                acc[2 * h] = __fadd_rn(acc[2 * h], __fmul_rn(coef[r], bf16_lo(w4[h])));
                                acc[2 * h + 1] =
                                    __fadd_rn(acc[2 * h + 1], __fmul_rn(coef[r], bf16_hi(w4[h])));
                            }
                        }
                    }
                    uint4 o;
                    o.x = pack_bf16x2(acc[0], acc[1]);
                    o.y = pack_bf16x2(acc[2], acc[3]);
                    o.z = pack_bf16x2(acc[4], acc[5]);
                    o.w = pack_bf16x2(acc[6], acc[7]);
                    reinterpret_cast<uint4*>(out)[j] = o;
                }
            }
        }
        cur = nxt;
    }
}

template <int MAXR, bool EXPERT>
cudaError_t launch_combine_t(const CombineArgs& a, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(a.P + 1) * 8;
    int per_sm = 0;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(combine_kernel<MAXR, EXPERT>), smem,
                                   kCombineThreads, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t warps_per_block = kCombineThreads / 32;
    const int64_t full_grid = static_cast<int64_t>(device_sm_count()) * per_sm;
    // Column halves only when whole tokens would take many rounds of the warps.
    const int split_shift = a.S >= kSplitRounds * full_grid * warps_per_block ? 1 : 0;
    int64_t grid = full_grid;
    const int64_t needed = ceil_div(a.S << split_shift, warps_per_block);
    if (grid > needed) grid = needed;
    return launch_pdl(combine_kernel<MAXR, EXPERT>, static_cast<unsigned>(grid), kCombineThreads, smem, stream, a,
                      split_shift);
}

template <bool EXPERT>
cudaError_t launch_combine_mode(const CombineArgs& a, int maxr, cudaStream_t stream) {
    if (a.S == 0) return cudaSuccess;
    if (maxr <= 1) return launch_combine_t<1, EXPERT>(a, stream);
    if (maxr <= 2) return launch_combine_t<2, EXPERT>(a, stream);
    if (maxr <= 4) return launch_combine_t<4, EXPERT>(a, stream);
    if (maxr <= 8) return launch_combine_t<8, EXPERT>(a, stream);
    return launch_combine_t<16, EXPERT>(a, stream);
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, CombineArgs a, cudaStream_t stream) {
    return launch_combine_mode<false>(a, s.K < s.P ? s.K : s.P, stream);  // distinct ranks of a token
}

cudaError_t launch_combine_expert(const moe_shape& s, CombineArgs a, cudaStream_t stream) {
    return launch_combine_mode<true>(a, s.K, stream);  // one row per slot
}

MOE_PROFILE_UNIT(combine)

}  // namespace moe
