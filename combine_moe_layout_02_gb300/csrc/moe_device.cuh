// moe_device.cuh -- device helpers shared by the sm_103a kernels of libmoe.so:
// mbarrier / bulk-copy (TMA) wrappers in inline PTX, warp utilities, and the
// launcher declarations the C-ABI layer calls.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// Upper bound on polls of one mbarrier phase before a kernel gives up, sets
// MOE_ERR_DEVICE_TIMEOUT and returns. try_wait itself suspends for a bounded
// time per poll, so this bounds the wait to seconds, far above any legitimate
// copy latency.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    return false;
}

// Global -> shared bulk copy; completion is counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global bulk copy, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte read-only load that skips L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch. Every kernel of the path is launched with
// programmatic stream serialisation: it may be scheduled while the previous
// kernel on the stream is still running. It waits for that kernel (and so,
// transitively, everything before it) to complete and flush before its first
// global-memory access, then lets the next kernel be scheduled.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Record a device-side status in the caller's error word (any writer wins;
// all writers of one launch write codes, never 0).
__device__ __forceinline__ void raise_error(int32_t* err, int32_t code) {
    if (err) *reinterpret_cast<volatile int32_t*>(err) = code;
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Balanced split of n items over b parts, the first n % b parts one larger.
__host__ __device__ __forceinline__ void split_range(int64_t n, int64_t b, int64_t i, int64_t* begin,
                                                     int64_t* end) {
    const int64_t q = n / b, r = n % b;
    const int64_t s = i * q + (i < r ? i : r);
    *begin = s;
    *end = s + q + (i < r ? 1 : 0);
}

// ---------------------------------------------------------------------------
// Launchers (defined in layout.cu / notify.cu / dispatch.cu / combine.cu).
// Shapes are validated by the C-ABI layer before these run.

struct LayoutPlan {
    int threads;       // tokens per block (one per thread)
    int64_t blocks_per_source;
    int64_t part_stride;  // int32 entries per block partial: P + E + 1
    size_t smem;
    int64_t scratch_bytes;
};
LayoutPlan layout_plan(const moe_shape& s);
cudaError_t launch_layout(const moe_shape& s, const int32_t* topk_idx, int32_t* ntpr, int32_t* ntpe,
                          uint8_t* itr, uint32_t* bits, int32_t* err, void* scratch,
                          cudaStream_t stream);

int64_t notify_scratch_bytes(const moe_shape& s);
cudaError_t launch_notify(const moe_shape& s, const int32_t* ntpr, const int32_t* ntpe,
                          const uint8_t* itr, int32_t* rpm, int32_t* cpm, int32_t* rcpm,
                          int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                          int64_t* part_row_base, void* scratch, cudaStream_t stream);

struct DispatchArgs {
    int32_t P, E, K, H, epr;
    int64_t S, T;
    const uint16_t* x;
    const int32_t* topk_idx;
    const float* topk_weights;
    const int32_t* send_head;
    const int64_t* part_row_base;
    uint8_t* arena;
    int64_t arena_rows;
    int64_t stride;
    int64_t scale_off;
    int64_t triple_off;
    int32_t* recv_src_idx;
    int32_t* recv_topk_idx;
    float* recv_topk_weights;
    int32_t* err;
    int32_t stages;
    uint32_t row_bytes;  // bf16 bytes of one source row, H * 2
    // Expert-major layout only: one slot per (token, k).
    const int32_t* slot_row;  // [S, K] row inside the destination rank's partition, or -1
    float* recv_weight;       // [rows] the slot's Top-K weight (may be NULL)
};
cudaError_t launch_dispatch(const moe_shape& s, DispatchArgs a, cudaStream_t stream);
cudaError_t launch_dispatch_expert(const moe_shape& s, DispatchArgs a, cudaStream_t stream);

struct CombineArgs {
    int32_t P, E, K, H, epr;
    int64_t S;
    const uint8_t* y;
    int64_t y_stride;
    const int64_t* part_row_base;
    int64_t arena_rows;
    const int32_t* send_head;
    const int32_t* topk_idx;
    const float* topk_weights;
    uint16_t* out;
    int32_t* err;
    const int32_t* slot_row;  // expert-major layout only
};
cudaError_t launch_combine(const moe_shape& s, CombineArgs a, cudaStream_t stream);
cudaError_t launch_combine_expert(const moe_shape& s, CombineArgs a, cudaStream_t stream);

int64_t notify_expert_scratch_bytes(const moe_shape& s);
cudaError_t launch_notify_expert(const moe_shape& s, const int32_t* topk_idx, const int32_t* nrtpe,
                                 const int32_t* reo, int32_t* slot_row, int64_t* expert_part_base,
                                 void* scratch, cudaStream_t stream);

cudaError_t launch_pad(const moe_shape& s, const int32_t* nrt, const int64_t* prb, uint8_t* arena,
                       int64_t arena_rows, int32_t* src_idx, int32_t* tk_idx, float* tk_w,
                       cudaStream_t stream);

bool fused_supported(const moe_shape& s);
int64_t fused_scratch_bytes(const moe_shape& s);
cudaError_t launch_fused(const moe_shape& s, const uint16_t* x, const int32_t* topk_idx, const float* topk_weights,
                         int32_t* ntpr, int32_t* ntpe, uint8_t* itr, uint32_t* bits, int32_t* rpm, int32_t* cpm,
                         int32_t* rcpm, int32_t* nrt, int32_t* nrtpe, int32_t* reo, int32_t* send_head,
                         int64_t* part_row_base, const DispatchArgs& d, int32_t* err, void* scratch,
                         cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Opt-in shared memory per block of the current device (cached).
int device_optin_smem();
// Shared memory of one SM (all its CTAs together), per current device.
int device_sm_smem();
// Allow `fn` `smem` bytes of dynamic shared memory on the current device and,
// if per_sm is given, return its resident blocks per SM for (threads, smem).
// Both are cached per (kernel, device).
cudaError_t prepare_kernel(const void* fn, size_t smem, int threads, int* per_sm);
// Static shared memory of `fn` (cached), or -1.
int kernel_static_smem(const void* fn);

// Launch `kernel` on `stream` with programmatic stream serialisation (see
// pdl_wait_then_release); the kernel must call pdl_wait_then_release before
// touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
