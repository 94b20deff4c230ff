/*
 * moe.h -- C ABI of libmoe.so, the GB300 (sm_103a) MoE dispatch/combine path.
 *
 * The path moves the hidden rows of S tokens to the expert-parallel ranks that
 * own their Top-K experts and reduces the experts' answers back:
 *
 *   moe_layout   topk_idx            -> per-rank / per-expert counts, token->rank table
 *   moe_notify   counts + table      -> prefix matrices, receive offsets, send_head
 *   moe_dispatch x + send_head       -> receive slots in P rank partitions (+ side arrays)
 *   moe_combine  expert rows (y)     -> out[S,H] = weighted sum over ranks
 *
 * The P expert-parallel ranks are P disjoint partitions of one receive arena
 * in this GPU's memory; "sending" a row to rank d means storing it in d's
 * partition. Source rank s owns global tokens [s*T, (s+1)*T), T = S / P.
 *
 * Problem statement followed ("Ascend DeepEP MoE Dispatch Optimization",
 * section "一条 token 如何走完 MoE"): inputs x[S,H], topk_idx[S,K],
 * topk_weights[S,K]; dst_rank = expert_id / experts_per_rank and
 * dst_local_expert = expert_id % experts_per_rank; one copy of the row per
 * distinct destination rank; combine returns the rows and reduces them by the
 * Top-K weights.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers, owned and allocated by the
 *     caller. The library never allocates device or pinned memory.
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns; results are ready when the stream
 *     reaches them. Nothing synchronises with the host.
 *   - The one exception to the two rules above is moe_run_host, the serving
 *     loop: it takes HOST buffers for the batches, uses its own streams and
 *     returns when the results are in host memory (see its declaration).
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED and enqueues
 *     nothing. MOE_ERR_CUDA means a launch failed.
 *   - Data-dependent problems (an expert id >= E, a receive row outside its
 *     partition or the arena, an inconsistent send_head) cannot be seen on the
 *     host. The kernels skip the offending element -- they never read or
 *     write out of bounds -- and store a moe_status code into the caller's
 *     device word `err` (may be NULL). moe_layout and moe_dispatch_fused
 *     always write `err` (0 or a code); the other calls only ever write a
 *     non-zero code into it.
 *   - Row-major layouts; int32 counts; the bf16 payload is passed as uint16
 *     bit patterns.
 *   - Alignment: every array pointer must be 16-byte aligned (the error word
 *     4-byte, scratch 256-byte); allocations from cudaMalloc or the PyTorch
 *     caching allocator are 256-byte aligned. y_row_stride is a multiple of 16.
 *   - Results are deterministic: the same inputs give the same bits on every
 *     run (no floating-point atomics, fixed reduction orders).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* bad pointer, size, alignment or shape      */
    MOE_ERR_TOPK_OUT_OF_RANGE = 2,  /* device: an expert id was >= E              */
    MOE_ERR_CAPACITY = 3,           /* device: a receive row fell outside its partition or the arena */
    MOE_ERR_CUDA = 4,               /* a CUDA launch or attribute call failed     */
    MOE_ERR_UNSUPPORTED = 5,        /* shape beyond the limits below              */
    MOE_ERR_DEVICE_TIMEOUT = 6,     /* device: a bounded wait on a copy gave up   */
    MOE_ERR_INCONSISTENT = 7        /* device: send_head names more ranks than the token's experts allow */
} moe_status;

/* Limits (the pages' CAM limits are P <= 384, E <= 512, K <= 16, H <= 7168). */
#define MOE_MAX_RANKS 1024
#define MOE_MAX_EXPERTS 4096
#define MOE_MAX_TOPK 16
#define MOE_MAX_HIDDEN 16384
/* Also S*K + E*(expert_alignment-1) <= INT32_MAX, so that every per-rank row
 * count and offset fits int32; larger shapes return MOE_ERR_UNSUPPORTED. */

/* Shape of one call. The tiling record of "HCCL Window 模式 (Non-SHMEM)
 * 代码深度剖析", section 8.1 (epWorldSize, moeExpertNum, quantMode, bs, k, h)
 * reduced to what the path needs. */
typedef struct moe_shape {
    int32_t P;                 /* expert-parallel ranks, 1..MOE_MAX_RANKS                  */
    int32_t E;                 /* experts, E % P == 0, P <= E <= MOE_MAX_EXPERTS            */
    int32_t S;                 /* global tokens, S % P == 0 (T = S / P per source rank), >= 0 */
    int32_t K;                 /* Top-K slots per token, 1..MOE_MAX_TOPK                    */
    int32_t H;                 /* hidden size, multiple of 8 (of 16 when quant = 1)          */
    int32_t num_channels;      /* C >= 1: shapes the channel prefix matrices only           */
    int32_t expert_alignment;  /* >= 1: per-expert receive counts are rounded up to it      */
    int32_t quant;             /* 0: bf16 payload; 1: int8 payload + fp32 scale             */
} moe_shape;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int32_t status);

/* Host-side check of a shape against the rules above. */
moe_status moe_check_shape(const moe_shape* shape);

/* Bytes per receive slot ("HCCL Window 模式 (Non-SHMEM) 代码深度剖析",
 * section 2.3 token format and section 8.2 size check):
 *   Ceil(Ceil(H * elt, 32) + 44, 512), elt = 2 (bf16) or 1 (int8).
 * Slot layout: payload [0, H*elt); fp32 scale at byte Ceil(H*elt, 32)
 * (int8 only; its 32-byte block is written, zero after the scale); int32
 * triple (source rank, source-local token, lowest k whose expert is on this
 * rank) at byte Ceil(H*elt, 32) + 32 (its 32-byte block is written, zero
 * after the triple); the rest is padding and is not written.
 * 14848 bytes for H = 7168 bf16. Returns -1 for H < 1. */
int64_t moe_slot_stride(int32_t H, int32_t quant);

/* Scratch bytes moe_layout, moe_notify, moe_notify_expert and
 * moe_dispatch_fused need for this shape (the calls may share one buffer; its
 * contents do not carry over between calls). */
int64_t moe_scratch_bytes(const moe_shape* shape);

/* Receive rows that always suffice when partitions are packed back to back
 * (part_row_base from moe_notify): S * min(K, P). */
int64_t moe_max_recv_rows(const moe_shape* shape);

/*
 * moe_layout -- the routing tables ("Ascend DeepEP MoE Dispatch
 * Optimization", sections "从 Python 接口进入真实调用链" and "Dispatch handle
 * 六项分别保存什么": num_tokens_per_rank, num_tokens_per_expert and the [S,P]
 * boolean is_token_in_rank).
 *
 *   topk_idx               int32 [S,K]  expert ids; any negative value is a
 *                                       masked slot; ids >= E are skipped and
 *                                       reported as MOE_ERR_TOPK_OUT_OF_RANGE
 *   num_tokens_per_rank    int32 [P,P]  [s][d] = tokens of source rank s with
 *                                       at least one expert on rank d
 *   num_tokens_per_expert  int32 [P,E]  [s][e] = slots of s's tokens equal to e
 *   is_token_in_rank       uint8 [S,P]  1 if token g has an expert on rank d
 *   is_token_in_rank_bits  uint32 [S,ceil(P/32)] or NULL: the same table packed,
 *                                       bit d%32 of word d/32
 *   err                    int32 device word or NULL; always written (0 or 2)
 *   scratch                >= moe_scratch_bytes(shape) bytes, 256-byte aligned
 */
moe_status moe_layout(const moe_shape* shape, const int32_t* topk_idx,
                      int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                      uint8_t* is_token_in_rank, uint32_t* is_token_in_rank_bits,
                      int32_t* err, void* scratch, int64_t scratch_bytes, void* stream);

/*
 * moe_notify -- counts and prefixes ("Ascend DeepEP MoE Dispatch
 * Optimization", section "Notify 先交换数量和前缀"; per-expert alignment from
 * "internode.cu", section 1 notify_dispatch; receive position from section
 * "Device 侧如何把 channel 变成远端 Put").
 *
 *   inputs: num_tokens_per_rank [P,P], num_tokens_per_expert [P,E],
 *           is_token_in_rank [S,P] (as written by moe_layout)
 *   rank_prefix_matrix         int32 [P,P]   [s][d] = sum over s' <= s of num_tokens_per_rank[s'][d]
 *   channel_prefix_matrix      int32 [P,P,C] [s][d][c] = tokens of s in channels 0..c bound for d
 *                                            (channel c = c-th block of the balanced split of T
 *                                            tokens over C, first T % C blocks one larger:
 *                                            "HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 8.3)
 *   recv_channel_prefix_matrix int32 [P,P,C] [d][s][c] = first row of (s, c)'s tokens in d's partition
 *   num_recv_tokens            int32 [P]     rows received by each rank
 *   num_recv_tokens_per_expert int32 [P,E/P] slots per local expert, rounded up to expert_alignment
 *   recv_expert_offset         int32 [P,E/P] exclusive scan of the line above, per rank
 *   send_head                  int32 [S,P]   row of token g inside d's partition, or -1 if not sent:
 *                                            rank_prefix[s-1][d] + channel_prefix[s][d][c-1] +
 *                                            running count inside the channel
 *   part_row_base              int64 [P+1]   exclusive scan of num_recv_tokens: partitions packed
 *                                            back to back; part_row_base[P] = total rows
 *   scratch                    >= moe_scratch_bytes(shape) bytes, 256-byte aligned
 */
moe_status moe_notify(const moe_shape* shape, const int32_t* num_tokens_per_rank,
                      const int32_t* num_tokens_per_expert, const uint8_t* is_token_in_rank,
                      int32_t* rank_prefix_matrix, int32_t* channel_prefix_matrix,
                      int32_t* recv_channel_prefix_matrix, int32_t* num_recv_tokens,
                      int32_t* num_recv_tokens_per_expert, int32_t* recv_expert_offset,
                      int32_t* send_head, int64_t* part_row_base,
                      void* scratch, int64_t scratch_bytes, void* stream);

/*
 * moe_dispatch -- the permutation ("HCCL Window 模式 (Non-SHMEM) 代码深度剖析",
 * section 3.6 InputToShare with the dynamic quantisation steps and FillTriple;
 * one copy per distinct rank as in "Ascend DeepEP MoE Dispatch Optimization").
 *
 * For every token g and rank d with send_head[g][d] >= 0, slot row
 * part_row_base[d] + send_head[g][d] of the arena receives:
 *   quant = 0: the bf16 row x[g], bit for bit;
 *   quant = 1: q[h] = clamp(rint(f32(x[g][h]) / scale), -127, 127) as int8 and
 *              scale = amax / 127 (binary32, round to nearest even; amax = max|x[g]|;
 *              amax == 0 gives scale 0 and q 0). Defined for finite x: a row with
 *              an infinity or NaN gets unspecified codes and scale (no error);
 *   the triple (g / T, g % T, lowest k with topk_idx[g][k] / (E/P) == d).
 * Side arrays (each may be NULL), indexed by arena row:
 *   recv_src_idx      int32 [arena_rows]    g % T
 *   recv_topk_idx     int32 [arena_rows,K]  topk_idx % (E/P) where the expert is on d, else -1
 *   recv_topk_weights float [arena_rows,K]  topk_weights where the expert is on d, else 0
 *
 *   x                bf16 bits [S,H], 16-byte aligned
 *   topk_idx         int32 [S,K]; topk_weights float [S,K] (may be NULL when
 *                    recv_topk_weights is NULL)
 *   part_row_base    int64 [P+1] device: first arena row of each partition;
 *                    moe_notify's packed bases, or any caller-chosen bases
 *                    (e.g. d * capacity for fixed-capacity partitions)
 *   recv_arena       arena_rows * moe_slot_stride(H, quant) bytes, 16-byte aligned
 *   err              int32 device word or NULL: rows outside [part_row_base[d],
 *                    part_row_base[d+1]) or beyond arena_rows are skipped and
 *                    raise MOE_ERR_CAPACITY
 */
moe_status moe_dispatch(const moe_shape* shape, const uint16_t* x, const int32_t* topk_idx,
                        const float* topk_weights, const int32_t* send_head,
                        const int64_t* part_row_base, void* recv_arena, int64_t arena_rows,
                        int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                        int32_t* err, void* stream);

/*
 * moe_combine -- the inverse permutation and weighted reduction ("HCCL Window
 * 模式 (Non-SHMEM) 代码深度剖析", section 7.8 ReadBufferAndWeightedSum: FP32
 * accumulator, Cast -> Muls -> Add per returned row, one CAST_RINT to BF16).
 *
 *   out[g][h] = bf16_rne( sum over d ascending with send_head[g][d] >= 0 of
 *                         c[g][d] * f32(y[part_row_base[d] + send_head[g][d]][h]) )
 *   c[g][d]   = sum, in ascending k, of topk_weights[g][k] over the slots whose
 *               expert is on d; 1 for every rank when topk_weights is NULL.
 * The accumulator starts at +0.0f; each product and each sum is rounded to
 * binary32 on its own (no fused multiply-add). A token with no valid rank
 * gives +0.
 *
 *   y             bf16 rows, y_row_stride bytes apart (a multiple of 16, >= 2H);
 *                 pass the dispatch arena with moe_slot_stride(H, 0) for
 *                 identity experts
 *   part_row_base int64 [P+1] device, as for moe_dispatch; arena_rows bounds the rows read
 *   send_head     int32 [S,P]; topk_idx int32 [S,K]; topk_weights float [S,K] or NULL
 *   out           bf16 bits [S,H], 16-byte aligned
 *   err           int32 device word or NULL (MOE_ERR_CAPACITY, MOE_ERR_INCONSISTENT)
 */
moe_status moe_combine(const moe_shape* shape, const void* y, int64_t y_row_stride,
                       const int64_t* part_row_base, int64_t arena_rows,
                       const int32_t* send_head, const int32_t* topk_idx,
                       const float* topk_weights, uint16_t* out, int32_t* err, void* stream);

/*
 * moe_dispatch_fused -- moe_layout + moe_notify + moe_dispatch in one launch,
 * for the small-message regime where the fixed cost of the routing tables
 * dominates the payload ("Ascend DeepEP MoE Dispatch Optimization", section
 * "128P 为什么会放大问题"; the single-kernel counting + prefix + copy shape of
 * "DeepEP Warp Specialization 深度分析", dispatch_impl). Every output has the
 * meaning, layout and value of the three separate calls with packed partitions
 * (part_row_base is written here and used for the rows).
 *
 * One cooperative persistent kernel (two CTAs per SM when their row buffers
 * fit in half an SM's shared memory, else one) with two bounded grid barriers;
 * the barrier counter lives in scratch and is zeroed by a one-thread kernel
 * launched on the stream just before. `err` is always written: cleared by the kernel, then
 * raised to MOE_ERR_TOPK_OUT_OF_RANGE, MOE_ERR_CAPACITY or
 * MOE_ERR_DEVICE_TIMEOUT if needed.
 * Supported: P <= 64, E <= 1024, H <= 8192, K <= 16, P * num_channels <= 4096,
 * quant = 0; other shapes return MOE_ERR_UNSUPPORTED (use the separate calls).
 * scratch >= moe_scratch_bytes.
 */
moe_status moe_dispatch_fused(const moe_shape* shape, const uint16_t* x, const int32_t* topk_idx,
                              const float* topk_weights, int32_t* num_tokens_per_rank,
                              int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                              uint32_t* is_token_in_rank_bits, int32_t* rank_prefix_matrix,
                              int32_t* channel_prefix_matrix, int32_t* recv_channel_prefix_matrix,
                              int32_t* num_recv_tokens, int32_t* num_recv_tokens_per_expert,
                              int32_t* recv_expert_offset, int32_t* send_head, int64_t* part_row_base,
                              void* recv_arena, int64_t arena_rows, int32_t* recv_src_idx,
                              int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* err, void* scratch,
                              int64_t scratch_bytes, void* stream);

/*
 * Expert-major receive layout ("HCCL Window 模式 (Non-SHMEM) 代码深度剖析",
 * section 3.6 InputToShare and section 7.8 ReadBufferAndWeightedSum). Instead of
 * one row per (token, destination rank), every valid (token, k) slot gets its
 * own row, and rank d's partition holds its experts' rows expert by expert:
 * local expert l starts at recv_expert_offset[d][l] (counts rounded up to
 * expert_alignment; rows in the alignment gaps are not written), and inside an
 * expert the slots are in (token, k) order. Each expert's rows are contiguous,
 * ready for a grouped expert GEMM.
 *
 * moe_max_expert_rows: arena rows that always suffice: S*K + E*(expert_alignment-1).
 *
 * moe_notify_expert -- after moe_layout and moe_notify:
 *   topk_idx                   int32 [S,K]
 *   num_recv_tokens_per_expert int32 [P,E/P] and recv_expert_offset int32 [P,E/P] from moe_notify
 *   slot_row                   int32 [S,K]   row of slot (g,k) inside rank (topk_idx/(E/P))'s
 *                                            partition: recv_expert_offset[e] + the number of
 *                                            earlier slots (token-major order) of expert e;
 *                                            -1 for a masked or out-of-range slot
 *   expert_part_base           int64 [P+1]   exclusive scan of the ranks' aligned row totals
 *   scratch                    >= moe_scratch_bytes(shape) bytes, 256-byte aligned
 *
 * moe_dispatch_expert -- for every valid slot, row expert_part_base[d] + slot_row[g][k]
 *   receives the payload (bf16, or int8 + scale, as moe_dispatch), the triple
 *   (g / T, g % T, k), recv_src_idx[row] = g % T and recv_weight[row] =
 *   topk_weights[g][k] (1 if topk_weights is NULL). Side arrays may be NULL.
 *   Rows outside their partition or the arena are skipped (MOE_ERR_CAPACITY in err).
 *
 * moe_combine_expert --
 *   out[g] = bf16_rne( sum over k ascending with a valid slot of
 *                      w[g][k] * f32(y[expert_part_base[d] + slot_row[g][k]]) )
 *   binary32 accumulator from +0, each product and sum rounded on its own, w = 1
 *   when topk_weights is NULL. y rows are y_row_stride bytes apart.
 */
int64_t moe_max_expert_rows(const moe_shape* shape);
moe_status moe_notify_expert(const moe_shape* shape, const int32_t* topk_idx,
                             const int32_t* num_recv_tokens_per_expert, const int32_t* recv_expert_offset,
                             int32_t* slot_row, int64_t* expert_part_base, void* scratch,
                             int64_t scratch_bytes, void* stream);
moe_status moe_dispatch_expert(const moe_shape* shape, const uint16_t* x, const int32_t* topk_idx,
                               const float* topk_weights, const int32_t* slot_row,
                               const int64_t* expert_part_base, void* recv_arena, int64_t arena_rows,
                               int32_t* recv_src_idx, float* recv_weight, int32_t* err, void* stream);
moe_status moe_combine_expert(const moe_shape* shape, const void* y, int64_t y_row_stride,
                              const int64_t* expert_part_base, int64_t arena_rows, const int32_t* slot_row,
                              const int32_t* topk_idx, const float* topk_weights, uint16_t* out,
                              int32_t* err, void* stream);

/*
 * moe_pad_partitions -- fixed-length receive partitions ("Ascend DeepEP MoE
 * Dispatch Optimization", section "输出长度有动态和固定两种模式": with a fixed
 * output length, num_worst_tokens, the host reads no count back and the rows
 * past the received count are padding -- x, scales and weights 0, topk_idx -1).
 *
 * With fixed-capacity partitions (part_row_base[d] = d * capacity, passed to
 * moe_dispatch) this fills, for every rank d, the rows from
 * part_row_base[d] + num_recv_tokens[d] up to part_row_base[d+1] (and below
 * arena_rows): payload 0, the scale block 0 (int8 slots), the triple
 * (-1, -1, -1), recv_src_idx -1, recv_topk_idx -1, recv_topk_weights 0 (each
 * side array may be NULL). A partition that overflowed (count > capacity) has
 * no padding; moe_dispatch reports the overflow rather than truncating.
 *
 *   num_recv_tokens int32 [P] (from moe_notify); part_row_base int64 [P+1];
 *   recv_arena / side arrays as for moe_dispatch. Only padding rows are written.
 */
moe_status moe_pad_partitions(const moe_shape* shape, const int32_t* num_recv_tokens,
                              const int64_t* part_row_base, void* recv_arena, int64_t arena_rows,
                              int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                              void* stream);

/*
 * moe_layout_static_scratch -- moe_layout without a caller-provided scratch
 * buffer. The pages have no counterpart: this entry point exists for callers
 * that cannot allocate device memory, such as code hosted by an engine that
 * owns all device memory and forbids allocation after start-up, or serving
 * loops where cudaMalloc would stall the device. Inputs, outputs and results
 * are those of moe_layout; the one scratch array moe_layout needs (an
 * out-of-range flag per source rank, folded into err) is a buffer of
 * MOE_LAYOUT_STATIC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits.
 *   - The buffer holds the flags of the largest shape moe_check_shape
 *     accepts (MOE_MAX_RANKS source ranks). A shape needing more is refused
 *     with MOE_ERR_UNSUPPORTED before anything is enqueued (moe_check_shape
 *     already refuses every such shape the same way).
 *   - The first call on each device looks up the buffer's device address
 *     (with that device current) and keeps it for the life of the process;
 *     make that first call before any stream capture. The kept address
 *     assumes the device's primary context is never reset or destroyed
 *     (cudaDeviceReset): after a reset, do not call this entry point again
 *     in the same process.
 *   - All calls share the buffer, which keeps the last call's contents;
 *     every flag is written before it is read, so nothing needs to start at
 *     zero. Calls that overlap on the GPU (different streams or threads)
 *     race on it: serialise them. Calls enqueued one after another on one
 *     stream are serialised by the stream.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define MOE_LAYOUT_STATIC_SCRATCH_BYTES (MOE_MAX_RANKS * 4u)
moe_status moe_layout_static_scratch(const moe_shape* shape, const int32_t* topk_idx,
                                     int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                                     uint8_t* is_token_in_rank, uint32_t* is_token_in_rank_bits,
                                     int32_t* err, void* stream);

/*
 * moe_run_host -- the whole path (moe_layout -> moe_notify -> moe_dispatch ->
 * moe_combine, or moe_dispatch_fused -> moe_combine) over n_batches batches
 * held in HOST memory, end to end: each batch's x, topk_idx and topk_weights
 * are copied to the device, routed, exchanged and reduced, and its combined
 * rows are copied back to out_host[i]. The pages have no single call for
 * this; it is the serving loop around the path ("Ascend DeepEP MoE Dispatch
 * Optimization", section "一条 token 如何走完 MoE": route, exchange, reduce,
 * per batch).
 *
 * Three internal streams overlap consecutive batches: while batch i computes,
 * batch i + 1's inputs are copied in and batch i - 1's output is copied out.
 * Inputs and outputs are double-buffered in the workspace; all other buffers
 * are used in batch order. The call is blocking: it first waits for all work
 * already submitted to the device, and returns when every copy has landed in
 * host memory. It is not capturable in a CUDA graph.
 *
 *   x_host[i]            bf16 bits [S,H] of batch i (pinned host memory for
 *                        copies that overlap; any host memory is accepted)
 *   topk_idx_host[i]     int32 [S,K]
 *   topk_weights_host    NULL (unit weights, as in moe_combine) or an array of
 *                        n_batches pointers to float [S,K]
 *   out_host[i]          bf16 bits [S,H], written with batch i's combine
 *                        result; entries may alias (batches are written back
 *                        in order)
 *   y, y_row_stride      expert outputs read by combine, device memory of at
 *                        least max(moe_max_recv_rows, moe_max_expert_rows)
 *                        rows; NULL means identity experts (combine reads the
 *                        bf16 dispatch arena, quant must be 0)
 *   flags                0 (rank-major layout), MOE_RUN_FUSED (use
 *                        moe_dispatch_fused when it supports the shape,
 *                        otherwise the separate calls) or MOE_RUN_EXPERT (the
 *                        expert-major layout: moe_notify_expert,
 *                        moe_dispatch_expert, moe_combine_expert); not both
 *   workspace            >= moe_run_host_workspace_bytes(shape, n_batches)
 *                        device bytes, 256-byte aligned, owned by the caller
 *   err_host             NULL or int32 [n_batches] host array: each batch's
 *                        device error word (0, or a moe_status code)
 * Returns MOE_OK, a host-side error (nothing run), MOE_ERR_CUDA, or the first
 * nonzero device error word in batch order.
 */
#define MOE_RUN_FUSED 1
#define MOE_RUN_EXPERT 2
int64_t moe_run_host_workspace_bytes(const moe_shape* shape, int32_t n_batches);
moe_status moe_run_host(const moe_shape* shape, int32_t n_batches, const uint16_t* const* x_host,
                        const int32_t* const* topk_idx_host, const float* const* topk_weights_host,
                        uint16_t* const* out_host, const void* y, int64_t y_row_stride, int32_t flags,
                        void* workspace, int64_t workspace_bytes, int32_t* err_host);

/*
 * moe_exchange_plan -- HOST function, for the path spread over P GPUs (one
 * expert-parallel rank each). After every rank has run moe_layout on its own
 * T tokens, the ranks all-gather their rows of num_tokens_per_rank and
 * num_tokens_per_expert ("internode.cu", section 1 notify_dispatch: counts
 * exchanged, then global prefix sums; "Ascend DeepEP MoE Dispatch
 * Optimization", section "Notify 先交换数量和前缀"). From the gathered tables
 * this computes what rank `self` needs before any row moves; every value is
 * the one moe_notify computes from the full tables.
 *
 *   ntpr_all [P,P], ntpe_all [P,E]   int32, host: row s = rank s's layout row
 *   rank_prefix_matrix [P,P]         int32, host (or NULL): inclusive column prefix
 *   num_recv_tokens [P]              int32, host (or NULL): rows each rank receives
 *   send_row_base [P]                int64, host (or NULL): first row of self's
 *                                    tokens inside rank d's receive partition
 *   self_recv_tokens_per_expert [E/P] int32, host (or NULL): self's experts'
 *                                    receive counts, rounded up to expert_alignment
 *   self_recv_expert_offset [E/P]    int32, host (or NULL): their exclusive scan
 *   part_row_base [P+1]              int64, host (or NULL): the packed bases of all
 *                                    partitions (the one-GPU emulation's layout)
 * Touches no device. Returns MOE_ERR_INVALID_ARG for a bad rank or a negative
 * count, MOE_ERR_UNSUPPORTED if a count overflows int32.
 */
moe_status moe_exchange_plan(const moe_shape* shape, int32_t self, const int32_t* ntpr_all,
                             const int32_t* ntpe_all, int32_t* rank_prefix_matrix, int32_t* num_recv_tokens,
                             int64_t* send_row_base, int32_t* self_recv_tokens_per_expert,
                             int32_t* self_recv_expert_offset, int64_t* part_row_base);

/*
 * moe_test_fused_barrier -- test hook for the bounded waits of
 * moe_dispatch_fused; the pages have no counterpart. It arms the NEXT
 * moe_dispatch_fused call made by this host thread (and that call only):
 * each of its grid barriers gives up after `spin_limit` polls (instead of
 * several million), and if skip_cta >= 0 the CTA with that index leaves out
 * its arrival at the first barrier. Every CTA's wait then runs out: the call
 * records MOE_ERR_DEVICE_TIMEOUT in err, each CTA waits (bounded) for its own
 * row loads to land and returns, and the context stays usable. It exists so
 * that tests can make a device-side wait time out without a fault. Returns
 * MOE_ERR_INVALID_ARG for spin_limit = 0.
 */
moe_status moe_test_fused_barrier(uint32_t spin_limit, int32_t skip_cta);

/*
 * moe_profile_attach -- profile builds only (compiled with -DMOE_PROFILE into
 * libmoe_profile.so; the default libmoe.so has no such symbol and its kernels
 * record nothing). The pages' "Ascend DeepEP MoE Dispatch Optimization",
 * section "Device 侧计时": per-core phase times written to exclusive slots
 * behind a compile-time switch that costs nothing when off.
 *
 * Points every instrumented kernel at `slots`, a device array of
 * MOE_PROF_KERNELS * MOE_PROF_CTAS * MOE_PROF_PHASES uint64 (bytes >= that
 * times 8, 16-byte aligned), or detaches them (slots = NULL). Thereafter CTA b
 * of kernel k writes row (k * MOE_PROF_CTAS + b) * MOE_PROF_PHASES:
 *   slot 0: %globaltimer (ns) when the CTA starts its work (after waiting for
 *           the previous kernel on the stream);
 *   slot p >= 1: the CTA's clock64 cycles from then to the end of phase p,
 *           or, for the int8 consumer's per-token steps, that step's cycles
 *           summed over the CTA's first consumer warp's tokens (added to:
 *           clear the array before a run).
 *   slot MOE_PROF_PHASES - 1: 1 + the SM the CTA ran on (%smid).
 * Kernel ids: 0 layout, 1 notify (either kernel), 2 dispatch bf16, 3 dispatch
 * int8, 4 combine, 5 fused, 6 notify_expert's rows kernel, 7 its count
 * kernel. CTAs at or beyond MOE_PROF_CTAS record nothing. Synchronous (a copy to each kernel unit's device pointer); call it
 * with no work of this library in flight. Outputs are unchanged.
 */
#define MOE_PROF_KERNELS 8
#define MOE_PROF_CTAS 4096
#define MOE_PROF_PHASES 16
#ifdef MOE_PROFILE
moe_status moe_profile_attach(void* slots, int64_t bytes);
#endif

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MOE_H_ */
