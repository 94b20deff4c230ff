// pad.cu -- padding of fixed-length receive partitions (moe_pad_partitions).
//
// "Ascend DeepEP MoE Dispatch Optimization", section "输出长度有动态和固定两种模式":
// when the caller fixes each rank's output length instead of reading the
// received count back, the rows past the count are padding: x, scales and
// weights 0, topk_idx -1. Here a partition of fixed capacity is
// [part_row_base[d], part_row_base[d+1]); its rows from
// part_row_base[d] + num_recv_tokens[d] on get a zero payload (and a zero
// scale block for int8 slots), the triple (-1, -1, -1), recv_src_idx -1,
// recv_topk_idx -1 and recv_topk_weights 0. A partition whose count exceeds
// its capacity has no padding (moe_dispatch reports the overflow).
//
// One block per (rank, row stripe); each row is cleared with 16-byte stores by
// the whole block. Only padding rows are touched.
#include "moe_device.cuh"

namespace moe {
namespace {

constexpr int kPadThreads = 256;
constexpr int kPadStripes = 16;

__global__ void __launch_bounds__(kPadThreads)
pad_kernel(int32_t P, int32_t K, int64_t payload_bytes, int64_t stride, int64_t scale_off,
           int64_t triple_off, bool quant, const int32_t* __restrict__ nrt,
           const int64_t* __restrict__ prb, uint8_t* __restrict__ arena, int64_t arena_rows,
           int32_t* __restrict__ src_idx, int32_t* __restrict__ tk_idx, float* __restrict__ tk_w) {
    pdl_wait_then_release();
    const int d = blockIdx.x / kPadStripes, stripe = blockIdx.x % kPadStripes;
    const int64_t lo = prb[d] + (nrt[d] > 0 ? static_cast<int64_t>(nrt[d]) : 0);
    int64_t hi = prb[d + 1];
    if (hi > arena_rows) hi = arena_rows;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (int64_t r = (lo > 0 ? lo : 0) + stripe; r < hi; r += kPadStripes) {
        uint8_t* slot = arena + r * stride;
        for (int64_t i = threadIdx.x; i < payload_bytes / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(slot)[i] = zero;
        if (threadIdx.x == 0) {
            if (quant) {
                reinterpret_cast<uint4*>(slot + scale_off)[0] = zero;
                reinterpret_cast<uint4*>(slot + scale_off)[1] = zero;
            }
            int4* t = reinterpret_cast<int4*>(slot + triple_off);
            t[0] = make_int4(-1, -1, -1, 0);
            t[1] = make_int4(0, 0, 0, 0);
            if (src_idx) src_idx[r] = -1;
        }
        for (int k = threadIdx.x; k < K; k += blockDim.x) {
            if (tk_idx) tk_idx[r * K + k] = -1;
            if (tk_w) tk_w[r * K + k] = 0.f;
        }
    }
}

}  // namespace

cudaError_t launch_pad(const moe_shape& s, const int32_t* nrt, const int64_t* prb, uint8_t* arena,
                       int64_t arena_rows, int32_t* src_idx, int32_t* tk_idx, float* tk_w,
                       cudaStream_t stream) {
    if (arena_rows == 0) return cudaSuccess;
    const int64_t elt = s.quant ? 1 : 2;
    const int64_t scale_off = round_up(static_cast<int64_t>(s.H) * elt, 32);
    const int64_t stride = round_up(scale_off + 44, 512);
    return launch_pdl(pad_kernel, static_cast<unsigned>(s.P) * kPadStripes, kPadThreads, 0, stream, s.P, s.K,
                      static_cast<int64_t>(s.H) * elt, stride, scale_off, scale_off + 32, s.quant != 0, nrt, prb,
                      arena, arena_rows, src_idx, tk_idx, tk_w);
}

}  // namespace moe
