// run.cu -- moe_run_host: the hot path over a sequence of batches held in
// host memory, end to end (host -> device copies, layout -> notify ->
// dispatch -> combine, device -> host copies).
//
// The path itself ("Ascend DeepEP MoE Dispatch Optimization", section
// "一条 token 如何走完 MoE": route, exchange, reduce) is enqueued through the
// public entry points; this file only stages data. Three streams overlap the
// stages of consecutive batches: while batch i computes, the inputs of batch
// i + 1 are copied in and the output of batch i - 1 is copied out. Inputs and
// outputs are double-buffered on the device; everything else (handle tensors,
// receive arena, scratch) is used by the compute stream only, in order.
//
//   H2D stream:     [wait compute(i-2)] copy x, topk_idx, topk_weights -> slot i%2, record h2d(i)
//   compute stream: [wait h2d(i), d2h(i-2)] layout, notify, dispatch, combine -> out slot i%2,
//                   record compute(i)   (or the expert-major calls, or fused -> combine)
//   D2H stream:     [wait compute(i)] copy out slot i%2 -> host, record d2h(i)
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "moe.h"

namespace {

constexpr int64_t kAlign = 256;

int64_t round_to(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Device buffers carved from one workspace. With base == nullptr only the
// size is computed.
struct RunBuffers {
    uint16_t* x[2];
    int32_t* idx[2];
    float* w[2];
    uint16_t* out[2];
    int32_t *ntpr, *ntpe, *rpm, *cpm, *rcpm, *nrt, *nrtpe, *reo, *send_head, *errs, *slot_row;
    uint8_t* itr;
    int64_t *prb, *expert_part_base;
    void* arena;
    void* scratch;
    int64_t arena_rows, scratch_bytes, total;
};

RunBuffers carve(const moe_shape& s, int64_t n_batches, unsigned char* base) {
    RunBuffers b{};
    int64_t off = 0;
    auto take = [&](int64_t bytes) -> void* {
        void* p = base ? static_cast<void*>(base + off) : nullptr;
        off += round_to(bytes > 0 ? bytes : 1, kAlign);
        return p;
    };
    const int64_t S = s.S, P = s.P, E = s.E, K = s.K, H = s.H, C = s.num_channels;
    for (int i = 0; i < 2; ++i) {
        b.x[i] = static_cast<uint16_t*>(take(S * H * 2));
        b.idx[i] = static_cast<int32_t*>(take(S * K * 4));
        b.w[i] = static_cast<float*>(take(S * K * 4));
        b.out[i] = static_cast<uint16_t*>(take(S * H * 2));
    }
    b.ntpr = static_cast<int32_t*>(take(P * P * 4));
    b.ntpe = static_cast<int32_t*>(take(P * E * 4));
    b.itr = static_cast<uint8_t*>(take(S * P));
    b.rpm = static_cast<int32_t*>(take(P * P * 4));
    b.cpm = static_cast<int32_t*>(take(P * P * C * 4));
    b.rcpm = static_cast<int32_t*>(take(P * P * C * 4));
    b.nrt = static_cast<int32_t*>(take(P * 4));
    b.nrtpe = static_cast<int32_t*>(take(E * 4));
    b.reo = static_cast<int32_t*>(take(E * 4));
    b.send_head = static_cast<int32_t*>(take(S * P * 4));
    b.prb = static_cast<int64_t*>(take((P + 1) * 8));
    b.slot_row = static_cast<int32_t*>(take(S * K * 4));
    b.expert_part_base = static_cast<int64_t*>(take((P + 1) * 8));
    // One arena for either layout: rank-major rows or expert-major slots.
    const int64_t rank_rows = moe_max_recv_rows(&s), expert_rows = moe_max_expert_rows(&s);
    b.arena_rows = rank_rows > expert_rows ? rank_rows : expert_rows;
    b.arena = take(b.arena_rows * moe_slot_stride(s.H, s.quant));
    b.scratch_bytes = moe_scratch_bytes(&s);
    b.scratch = take(b.scratch_bytes);
    b.errs = static_cast<int32_t*>(take(n_batches * 4));
    b.total = off;
    return b;
}

// Streams and events of one call, released on every path.
struct Pipeline {
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t h2d_done[2] = {nullptr, nullptr}, comp_done[2] = {nullptr, nullptr},
                d2h_done[2] = {nullptr, nullptr};
    cudaError_t init() {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&comp, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (int i = 0; i < 2; ++i) {
            if ((e = cudaEventCreateWithFlags(&h2d_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&comp_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&d2h_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    ~Pipeline() {
        for (cudaStream_t s : {h2d, comp, d2h})
            if (s) cudaStreamSynchronize(s);
        for (int i = 0; i < 2; ++i) {
            if (h2d_done[i]) cudaEventDestroy(h2d_done[i]);
            if (comp_done[i]) cudaEventDestroy(comp_done[i]);
            if (d2h_done[i]) cudaEventDestroy(d2h_done[i]);
        }
        for (cudaStream_t s : {h2d, comp, d2h})
            if (s) cudaStreamDestroy(s);
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int64_t moe_run_host_workspace_bytes(const moe_shape* shape, int32_t n_batches) {
    if (moe_check_shape(shape) != MOE_OK || n_batches < 0) return -1;
    return carve(*shape, n_batches, nullptr).total;
}

moe_status moe_run_host(const moe_shape* shape, int32_t n_batches, const uint16_t* const* x_host,
                        const int32_t* const* topk_idx_host, const float* const* topk_weights_host,
                        uint16_t* const* out_host, const void* y, int64_t y_row_stride, int32_t flags,
                        void* workspace, int64_t workspace_bytes, int32_t* err_host) {
    moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const moe_shape& s = *shape;
    if (n_batches < 0 || (flags & ~(MOE_RUN_FUSED | MOE_RUN_EXPERT)) != 0) return MOE_ERR_INVALID_ARG;
    // The fused launch builds the rank-major layout only.
    if ((flags & MOE_RUN_FUSED) && (flags & MOE_RUN_EXPERT)) return MOE_ERR_INVALID_ARG;
    if (n_batches == 0) return MOE_OK;
    if (!x_host || !topk_idx_host || !out_host || !workspace || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return MOE_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_batches; ++i) {
        if (s.S > 0 && (!x_host[i] || !topk_idx_host[i] || !out_host[i])) return MOE_ERR_INVALID_ARG;
        if (topk_weights_host && s.S > 0 && !topk_weights_host[i]) return MOE_ERR_INVALID_ARG;
    }
    // Combine reads the expert outputs y; without them (identity experts) it
    // reads the dispatch arena, which holds bf16 rows only.
    if (!y && s.quant != 0) return MOE_ERR_INVALID_ARG;
    // y as moe_combine checks it, here before anything is enqueued.
    if (y && (!aligned16(y) || y_row_stride < 2 * static_cast<int64_t>(s.H) || y_row_stride % 16 != 0))
        return MOE_ERR_INVALID_ARG;
    const RunBuffers b = carve(s, n_batches, static_cast<unsigned char*>(workspace));
    if (workspace_bytes < b.total) return MOE_ERR_INVALID_ARG;
    const void* yy = y ? y : b.arena;
    const int64_t ys = y ? y_row_stride : moe_slot_stride(s.H, 0);
    const int64_t S = s.S, H = s.H, K = s.K;
    const bool weights = topk_weights_host != nullptr;

    // Earlier work on the device may still use the workspace or the host buffers.
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    Pipeline pl;
    if (pl.init() != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(b.errs, 0, static_cast<size_t>(n_batches) * 4, pl.comp) != cudaSuccess) return MOE_ERR_CUDA;
    bool fused = (flags & MOE_RUN_FUSED) != 0;
    const bool expert = (flags & MOE_RUN_EXPERT) != 0;

    for (int32_t i = 0; i < n_batches; ++i) {
        const int sl = i & 1;
        // inputs of batch i into slot sl, once batch i - 2 no longer reads it
        if (i >= 2 && cudaStreamWaitEvent(pl.h2d, pl.comp_done[sl], 0) != cudaSuccess) return MOE_ERR_CUDA;
        if (S > 0) {
            if (cudaMemcpyAsync(b.x[sl], x_host[i], S * H * 2, cudaMemcpyHostToDevice, pl.h2d) != cudaSuccess ||
                cudaMemcpyAsync(b.idx[sl], topk_idx_host[i], S * K * 4, cudaMemcpyHostToDevice, pl.h2d) !=
                    cudaSuccess)
                return MOE_ERR_CUDA;
            if (weights && cudaMemcpyAsync(b.w[sl], topk_weights_host[i], S * K * 4, cudaMemcpyHostToDevice,
                                           pl.h2d) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        if (cudaEventRecord(pl.h2d_done[sl], pl.h2d) != cudaSuccess) return MOE_ERR_CUDA;

        // the path, once the inputs are in and out slot sl has been read back
        if (cudaStreamWaitEvent(pl.comp, pl.h2d_done[sl], 0) != cudaSuccess) return MOE_ERR_CUDA;
        if (i >= 2 && cudaStreamWaitEvent(pl.comp, pl.d2h_done[sl], 0) != cudaSuccess) return MOE_ERR_CUDA;
        const float* w = weights ? b.w[sl] : nullptr;
        int32_t* err = b.errs + i;
        if (fused) {
            st = moe_dispatch_fused(&s, b.x[sl], b.idx[sl], w, b.ntpr, b.ntpe, b.itr, nullptr, b.rpm, b.cpm,
                                    b.rcpm, b.nrt, b.nrtpe, b.reo, b.send_head, b.prb, b.arena, b.arena_rows,
                                    nullptr, nullptr, nullptr, err, b.scratch, b.scratch_bytes, pl.comp);
            if (st == MOE_ERR_UNSUPPORTED) fused = false;  // nothing was enqueued
            else if (st != MOE_OK) return st;
        }
        if (!fused) {
            st = moe_layout(&s, b.idx[sl], b.ntpr, b.ntpe, b.itr, nullptr, err, b.scratch, b.scratch_bytes,
                            pl.comp);
            if (st != MOE_OK) return st;
            st = moe_notify(&s, b.ntpr, b.ntpe, b.itr, b.rpm, b.cpm, b.rcpm, b.nrt, b.nrtpe, b.reo, b.send_head,
                            b.prb, b.scratch, b.scratch_bytes, pl.comp);
            if (st != MOE_OK) return st;
            if (expert) {
                st = moe_notify_expert(&s, b.idx[sl], b.nrtpe, b.reo, b.slot_row, b.expert_part_base, b.scratch,
                                       b.scratch_bytes, pl.comp);
                if (st != MOE_OK) return st;
                st = moe_dispatch_expert(&s, b.x[sl], b.idx[sl], w, b.slot_row, b.expert_part_base, b.arena,
                                         b.arena_rows, nullptr, nullptr, err, pl.comp);
            } else {
                st = moe_dispatch(&s, b.x[sl], b.idx[sl], w, b.send_head, b.prb, b.arena, b.arena_rows, nullptr,
                                  nullptr, nullptr, err, pl.comp);
            }
            if (st != MOE_OK) return st;
        }
        if (expert)
            st = moe_combine_expert(&s, yy, ys, b.expert_part_base, b.arena_rows, b.slot_row, b.idx[sl], w,
                                    b.out[sl], err, pl.comp);
        else
            st = moe_combine(&s, yy, ys, b.prb, b.arena_rows, b.send_head, b.idx[sl], w, b.out[sl], err, pl.comp);
        if (st != MOE_OK) return st;
        if (cudaEventRecord(pl.comp_done[sl], pl.comp) != cudaSuccess) return MOE_ERR_CUDA;

        // output of batch i back to the host
        if (cudaStreamWaitEvent(pl.d2h, pl.comp_done[sl], 0) != cudaSuccess) return MOE_ERR_CUDA;
        if (S > 0 && cudaMemcpyAsync(out_host[i], b.out[sl], S * H * 2, cudaMemcpyDeviceToHost, pl.d2h) !=
                         cudaSuccess)
            return MOE_ERR_CUDA;
        if (cudaEventRecord(pl.d2h_done[sl], pl.d2h) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (cudaStreamSynchronize(pl.d2h) != cudaSuccess || cudaStreamSynchronize(pl.comp) != cudaSuccess ||
        cudaStreamSynchronize(pl.h2d) != cudaSuccess)
        return MOE_ERR_CUDA;
    std::vector<int32_t> errs(static_cast<size_t>(n_batches));
    if (cudaMemcpy(errs.data(), b.errs, errs.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status first = MOE_OK;
    for (int32_t i = 0; i < n_batches; ++i) {
        if (err_host) err_host[i] = errs[static_cast<size_t>(i)];
        if (first == MOE_OK && errs[static_cast<size_t>(i)] != 0) first = static_cast<moe_status>(errs[static_cast<size_t>(i)]);
    }
    return first;
}

}  // extern "C"
