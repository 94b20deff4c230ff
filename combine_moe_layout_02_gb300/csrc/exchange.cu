// exchange.cu -- host-side plan of a multi-GPU exchange (moe_exchange_plan).
//
// On P GPUs each expert-parallel rank runs moe_layout on its own T tokens and
// holds only its row of num_tokens_per_rank and num_tokens_per_expert. Before
// any row moves, the ranks exchange those rows (an all-gather of P * (P + E)
// int32: "internode.cu", section 1, notify_dispatch -- per-rank and
// per-expert counts are exchanged, then every rank computes the global
// prefix sums it needs; "Ascend DeepEP MoE Dispatch Optimization", section
// "Notify 先交换数量和前缀"). From the gathered counts this function computes,
// on the host, what rank `self` needs:
//   - rank_prefix_matrix [P,P] and num_recv_tokens [P] (the column sums);
//   - send_row_base [P]: the first row of self's tokens inside each rank d's
//     receive partition, rank_prefix_matrix[self-1][d] (0 for self = 0) --
//     where self writes (or sends) its rows for d;
//   - self's aligned per-expert receive counts and their exclusive scan
//     (num_recv_tokens_per_expert / recv_expert_offset rows of rank self);
//   - part_row_base [P+1]: the packed bases of all partitions, the layout of
//     the one-GPU emulation in which rank d's partition is one slice of one
//     arena (what moe_notify computes on the device).
// Every value equals what moe_notify computes from the full tables.
#include <stdint.h>

#include "moe.h"

extern "C" moe_status moe_exchange_plan(const moe_shape* shape, int32_t self, const int32_t* ntpr_all,
                                        const int32_t* ntpe_all, int32_t* rank_prefix_matrix,
                                        int32_t* num_recv_tokens, int64_t* send_row_base,
                                        int32_t* self_recv_tokens_per_expert, int32_t* self_recv_expert_offset,
                                        int64_t* part_row_base) {
    const moe_status st = moe_check_shape(shape);
    if (st != MOE_OK) return st;
    const int32_t P = shape->P, E = shape->E, A = shape->expert_alignment;
    if (self < 0 || self >= P || !ntpr_all || !ntpe_all) return MOE_ERR_INVALID_ARG;
    const int32_t epr = E / P;
    // Column prefix over the source ranks, in rank order.
    for (int32_t d = 0; d < P; ++d) {
        int64_t run = 0;
        for (int32_t s = 0; s < P; ++s) {
            const int32_t v = ntpr_all[static_cast<int64_t>(s) * P + d];
            if (v < 0) return MOE_ERR_INVALID_ARG;
            if (send_row_base && s == self) send_row_base[d] = run;
            run += v;
            if (run > INT32_MAX) return MOE_ERR_UNSUPPORTED;
            if (rank_prefix_matrix) rank_prefix_matrix[static_cast<int64_t>(s) * P + d] = static_cast<int32_t>(run);
        }
        if (num_recv_tokens) num_recv_tokens[d] = static_cast<int32_t>(run);
    }
    // Rank self's experts: receive counts rounded up to the alignment, and
    // their exclusive scan.
    int64_t off = 0;
    for (int32_t l = 0; l < epr; ++l) {
        int64_t c = 0;
        for (int32_t s = 0; s < P; ++s) {
            const int32_t v = ntpe_all[static_cast<int64_t>(s) * E + static_cast<int64_t>(self) * epr + l];
            if (v < 0) return MOE_ERR_INVALID_ARG;
            c += v;
        }
        c = (c + A - 1) / A * A;
        if (c > INT32_MAX || off > INT32_MAX) return MOE_ERR_UNSUPPORTED;
        if (self_recv_tokens_per_expert) self_recv_tokens_per_expert[l] = static_cast<int32_t>(c);
        if (self_recv_expert_offset) self_recv_expert_offset[l] = static_cast<int32_t>(off);
        off += c;
    }
    // Packed bases of all partitions (the one-GPU emulation).
    if (part_row_base) {
        int64_t base = 0;
        for (int32_t d = 0; d < P; ++d) {
            part_row_base[d] = base;
            int64_t n = 0;
            for (int32_t s = 0; s < P; ++s) n += ntpr_all[static_cast<int64_t>(s) * P + d];
            base += n;
        }
        part_row_base[P] = base;
    }
    return MOE_OK;
}
