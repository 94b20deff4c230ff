// layout_static.cu -- moe_layout for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: code hosted inside an
// engine that owns every byte of device memory and forbids allocation once it
// has started, and latency-bound serving loops where an allocation would
// synchronise the device. moe_layout needs a scratch array (one out-of-range
// flag per source rank, folded into the error word by its tail kernel); this
// entry point takes it from a buffer compiled into the library instead, so
// the caller passes only the inputs and outputs.
//
// The buffer is a file-scope __device__ array of MOE_LAYOUT_STATIC_SCRATCH_BYTES
// bytes, enough for the largest accepted shape. Every GPU that loads the
// library holds it until the process exits. Host code cannot use the array's
// name as a device address, so the first call on each device looks the
// address up with cudaGetSymbolAddress (with that device current) and keeps
// it; that first call should therefore come before any stream capture, and
// the kept address assumes the device's context is never reset. All calls
// share the one buffer and it keeps the last call's contents: the layout
// kernel writes every flag before the tail kernel reads it, so nothing has to
// start at zero, but calls that overlap on the GPU (on two streams, or from
// two threads) race on it. Nothing here calls cudaMalloc, cudaFree or any
// routine that allocates.
#include <mutex>

#include "moe.h"
#include "moe_device.cuh"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_layout_scratch[MOE_LAYOUT_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of g_layout_scratch on the current device (resolved once).
cudaError_t static_scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status moe_layout_static_scratch(const moe_shape* shape, const int32_t* topk_idx,
                                                int32_t* num_tokens_per_rank,
                                                int32_t* num_tokens_per_expert,
                                                uint8_t* is_token_in_rank,
                                                uint32_t* is_token_in_rank_bits, int32_t* err,
                                                void* stream) {
    using namespace moe;
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    const int64_t S = s.S;
    if ((S > 0 && (!topk_idx || !is_token_in_rank)) || !num_tokens_per_rank || !num_tokens_per_expert)
        return MOE_ERR_INVALID_ARG;
    if ((topk_idx && !aligned16(topk_idx)) || (is_token_in_rank && !aligned16(is_token_in_rank)) ||
        !aligned16(num_tokens_per_rank) || !aligned16(num_tokens_per_expert) ||
        (is_token_in_rank_bits && !aligned16(is_token_in_rank_bits)) ||
        (err && (reinterpret_cast<uintptr_t>(err) & 3u)))
        return MOE_ERR_INVALID_ARG;
    // The flags of this shape must fit in the built-in buffer.
    if (layout_plan(s).scratch_bytes > static_cast<int64_t>(MOE_LAYOUT_STATIC_SCRATCH_BYTES))
        return MOE_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (static_scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t e = launch_layout(s, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                                  is_token_in_rank, is_token_in_rank_bits, err, scratch,
                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
