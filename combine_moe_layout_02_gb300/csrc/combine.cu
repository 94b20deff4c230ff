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
// Design (sm_103a): persistent grid, one CTA per token at a time. Warp 0 turns
// the token's send_head row into a compact list of (row address, weight) in
// ascending rank order (ballot + popc compaction). Then every thread owns
// 16-byte column chunks: it issues the loads of that chunk from all of the
// token's rows before reducing them, so up to MAXR x 16 bytes per thread are in
// flight, and writes one 16-byte chunk of out.
#include <cuda_bf16.h>

#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Two binary32 values to two bf16 (round to nearest even), packed low/high.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

template <int MAXR>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    extern __shared__ __align__(16) int64_t prb[];  // [P+1]
    __shared__ const uint8_t* s_row[MAXR];
    __shared__ float s_coef[MAXR];
    __shared__ int s_n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i <= a.P; i += blockDim.x) prb[i] = a.part_row_base[i];
    __syncthreads();
    const int nchunks = a.H / 8;
    const int K = a.K;
    for (int64_t g = blockIdx.x; g < a.S; g += gridDim.x) {
        if (warp == 0) {
            int32_t dk = -1;
            float w = 0.f;
            if (lane < K) {
                const int32_t idx = __ldg(a.topk_idx + g * K + lane);
                dk = (idx >= 0 && idx < a.E) ? idx / a.epr : -1;
                if (a.topk_weights) w = __ldg(a.topk_weights + g * K + lane);
            }
            int n = 0;
            for (int d0 = 0; d0 < a.P; d0 += 32) {
                const int d = d0 + lane;
                const int32_t sh = d < a.P ? __ldg(a.send_head + g * a.P + d) : -1;
                bool valid = false;
                int64_t row = 0;
                if (sh >= 0) {
                    const int64_t lo = prb[d], hi = prb[d + 1];
                    row = lo + sh;
                    valid = sh < hi - lo && row >= 0 && row < a.arena_rows;
                    if (!valid) raise_error(a.err, MOE_ERR_CAPACITY);
                }
                float c = 0.f;
                for (int k = 0; k < K; ++k) {
                    const int32_t dkk = __shfl_sync(0xffffffffu, dk, k);
                    const float wk = __shfl_sync(0xffffffffu, w, k);
                    if (dkk == d) c = __fadd_rn(c, wk);
                }
                if (!a.topk_weights) c = 1.f;
                const uint32_t bal = __ballot_sync(0xffffffffu, valid);
                if (valid) {
                    const int pos = n + __popc(bal & lanemask_lt());
                    if (pos < MAXR) {
                        s_row[pos] = a.y + row * a.y_stride;
                        s_coef[pos] = c;
                    } else {
                        raise_error(a.err, MOE_ERR_INCONSISTENT);
                    }
                }
                n += __popc(bal);
            }
            if (lane == 0) s_n = n < MAXR ? n : MAXR;
        }
        __syncthreads();
        const int n = s_n;
        uint16_t* out = a.out + g * a.H;
        for (int j = tid; j < nchunks; j += blockDim.x) {
            uint4 v[MAXR];
#pragma unroll
            for (int r = 0; r < MAXR; ++r)
                if (r < n) v[r] = ld_stream_u4(s_row[r] + static_cast<size_t>(j) * 16);
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
            for (int r = 0; r < MAXR; ++r) {
                if (r < n) {
                    const float c = s_coef[r];
                    const uint32_t u[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(c, bf16_lo(u[q])));
                        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(c, bf16_hi(u[q])));
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
        __syncthreads();
    }
}

template <int MAXR>
cudaError_t launch_combine_t(const CombineArgs& a, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(a.P + 1) * 8;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<MAXR>,
                                                                  kCombineThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = static_cast<int64_t>(device_sm_count()) * per_sm;
    if (grid > a.S) grid = a.S;
    combine_kernel<MAXR><<<static_cast<unsigned>(grid), kCombineThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const moe_shape& s, CombineArgs a, cudaStream_t stream) {
    if (a.S == 0) return cudaSuccess;
    const int maxr = s.K < s.P ? s.K : s.P;  // distinct ranks of one token
    if (maxr <= 1) return launch_combine_t<1>(a, stream);
    if (maxr <= 2) return launch_combine_t<2>(a, stream);
    if (maxr <= 4) return launch_combine_t<4>(a, stream);
    if (maxr <= 8) return launch_combine_t<8>(a, stream);
    return launch_combine_t<16>(a, stream);
}

}  // namespace moe
