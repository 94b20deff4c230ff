// moe_oracle.cpp -- CPU oracle for the MoE dispatch/combine hot path.
//
// TEST INFRASTRUCTURE ONLY. This file is the reference that the CUDA path is
// checked against. Only the tests, the smoke check and the CPU-baseline leg of
// the benchmark load it; the library under combine_moe_layout_02_gb300/ never
// does. It shares no header, helper, table or constant with the CUDA sources.
//
// Plain, single-threaded, slow on purpose: every output is computed by the
// loop that defines it, in global token order, with no blocking or fusion.
// Built with -O2 -ffp-contract=off so that a*b+c is never fused.
//
// Sources (page title, then section):
//   [R]  "Ascend DeepEP MoE Dispatch Optimization", section
//        "一条 token 如何走完 MoE": dst_rank = expert_id / experts_per_rank,
//        one copy of the hidden row per distinct destination rank, combine
//        reduces the returned rows by the Top-K weights.
//   [H]  same page, section "Dispatch handle 六项分别保存什么": the handle
//        tensors (rank_prefix_matrix, channel_prefix_matrix,
//        recv_channel_prefix_matrix, recv_src_idx, is_token_in_rank [S,P],
//        send_head [S,P] with -1 meaning "not sent to this rank").
//   [N]  same page, section "Notify 先交换数量和前缀": notify turns routing
//        into per-rank / per-expert counts and (source rank, channel) prefixes.
//   [D]  same page, section "Device 侧如何把 channel 变成远端 Put": a row's
//        receive position = rank prefix of the previous source rank + channel
//        prefix of the previous channel + running count inside the channel.
//   [A]  "internode.cu", section 1 "notify_dispatch": per-expert receive
//        counts are rounded up to a multiple of expert_alignment.
//   [F]  "HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 2.3 (token slot:
//        payload, pad to 32 B, fp32 dynamic scale, int32 triple
//        (rank, token, topk), pad to 512 B) and section 8.2 (slot size
//        Ceil(Ceil(h*elt,32)+44, 512)).
//   [S]  same page, section 8.3: balanced split of n items over b workers,
//        the first n % b workers take one extra item.
//   [Q]  same page, section 3.6: dynamic quantisation
//        BF16 -> FP32 -> Abs -> ReduceMax -> Scale -> INT8.
//   [C]  same page, section 7.8: FP32 accumulator; for each returned row
//        Cast to FP32, multiply by the weight, add; one final CAST_RINT to BF16.
//
// Readings where the pages leave a step open (each is also listed in the
// design notes of the repository):
//   * one copy per distinct destination rank (not per (token, k));
//   * negative expert ids are masked slots; ids >= E are errors (skipped);
//   * per-rank combine weight c_{g,d} = sum, in ascending k, of the weights of
//     the token's slots whose expert lives on d; NULL weights mean c = 1;
//   * ranks are reduced in ascending order, multiply and add rounded
//     separately (no fused multiply-add);
//   * scale = amax / 127 (binary32 division), q = rint(x / scale) (binary32
//     division, round-half-even), clamped to [-127, 127]; amax == 0 gives
//     scale 0 and q 0; the scale sits at byte Ceil(H*elt, 32) of the slot and
//     the triple 32 bytes after it;
//   * the triple's topk field is the lowest k whose expert lives on the
//     destination rank; recv_src_idx is the token index local to its source;
//   * send_head[g][d] is the row of token g inside rank d's receive
//     partition, or -1;
//   * channel c of a source rank owns the c-th block of the balanced split of
//     its T tokens over C channels; channel_prefix_matrix is inclusive over
//     channels, recv_channel_prefix_matrix holds exclusive start rows.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// --- bf16 <-> fp32, written out from the IEEE-754 binary32 layout ----------
float bf16_bits_to_float(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

// Round a binary32 value to the nearest bfloat16, ties to even ("RINT").
uint16_t float_to_bf16_bits_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u) {
        return static_cast<uint16_t>((u >> 16) | 0x0040u);  // quiet NaN
    }
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return static_cast<uint16_t>(keep);
}

int64_t ceil_to(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Channel c of a source rank with T tokens split over C channels: [S].
void channel_range(int64_t T, int64_t C, int64_t c, int64_t* begin, int64_t* end) {
    int64_t n = T / C;
    int64_t r = T % C;
    int64_t b = c * n + (c < r ? c : r);
    *begin = b;
    *end = b + n + (c < r ? 1 : 0);
}

// Is slot value idx a valid expert of rank d?
bool slot_on_rank(int32_t idx, int32_t E, int32_t epr, int32_t d) {
    return idx >= 0 && idx < E && idx / epr == d;
}

}  // namespace

extern "C" {

// Receive-slot size in bytes: [F] section 8.2.
int64_t oracle_slot_stride(int32_t H, int32_t quant) {
    int64_t elt = quant ? 1 : 2;
    int64_t payload = ceil_to(static_cast<int64_t>(H) * elt, 32);
    return ceil_to(payload + 44, 512);
}

// Layout [R][H]: per-source-rank counts and the token -> rank table.
//   num_tokens_per_rank  [P][P]  tokens of source s with >= 1 expert on d
//   num_tokens_per_expert[P][E]  slots of source s's tokens equal to e
//   is_token_in_rank     [S][P]  0/1
//   bits                 [S][ceil(P/32)] bit d%32 of word d/32 (may be NULL)
// Returns 0, or 2 when some expert id is >= E (those slots are skipped).
int32_t oracle_layout(int32_t P, int32_t E, int64_t S, int32_t K,
                      const int32_t* topk_idx,
                      int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                      uint8_t* is_token_in_rank, uint32_t* bits) {
    const int32_t epr = E / P;
    const int64_t T = S / P;
    const int32_t W = (P + 31) / 32;
    std::memset(num_tokens_per_rank, 0, sizeof(int32_t) * P * P);
    std::memset(num_tokens_per_expert, 0, sizeof(int32_t) * P * E);
    std::memset(is_token_in_rank, 0, static_cast<size_t>(S) * P);
    if (bits) std::memset(bits, 0, sizeof(uint32_t) * static_cast<size_t>(S) * W);
    int32_t err = 0;
    std::vector<uint8_t> seen(P);
    for (int64_t g = 0; g < S; ++g) {
        const int64_t s = g / T;
        std::fill(seen.begin(), seen.end(), 0);
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[g * K + k];
            if (e < 0) continue;                 // masked slot
            if (e >= E) { err = 2; continue; }   // out of range: report, skip
            num_tokens_per_expert[s * E + e] += 1;
            seen[e / epr] = 1;
        }
        for (int32_t d = 0; d < P; ++d) {
            if (!seen[d]) continue;
            is_token_in_rank[g * P + d] = 1;
            num_tokens_per_rank[s * P + d] += 1;
            if (bits) bits[g * W + d / 32] |= (1u << (d % 32));
        }
    }
    return err;
}

// Notify [N][H][D][A]. Outputs:
//   rank_prefix_matrix        [P][P]    inclusive over source ranks
//   channel_prefix_matrix     [P][P][C] inclusive over channels, per (s, d)
//   recv_channel_prefix_matrix[P][P][C] exclusive start row of (s, c) in d
//   num_recv_tokens           [P]
//   num_recv_tokens_per_expert[P][E/P]  rounded up to expert_alignment
//   recv_expert_offset        [P][E/P]  exclusive scan of the line above
//   send_head                 [S][P]    row inside d's partition, or -1
//   part_row_base             [P+1]     exclusive scan of num_recv_tokens
void oracle_notify(int32_t P, int32_t E, int64_t S, int32_t C, int32_t expert_alignment,
                   const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                   const uint8_t* is_token_in_rank,
                   int32_t* rank_prefix_matrix, int32_t* channel_prefix_matrix,
                   int32_t* recv_channel_prefix_matrix, int32_t* num_recv_tokens,
                   int32_t* num_recv_tokens_per_expert, int32_t* recv_expert_offset,
                   int32_t* send_head, int64_t* part_row_base) {
    const int32_t epr = E / P;
    const int64_t T = S / P;
    // Rank prefix: running sum down each destination column.
    for (int32_t d = 0; d < P; ++d) {
        int32_t run = 0;
        for (int32_t s = 0; s < P; ++s) {
            run += num_tokens_per_rank[s * P + d];
            rank_prefix_matrix[s * P + d] = run;
        }
        num_recv_tokens[d] = run;
    }
    part_row_base[0] = 0;
    for (int32_t d = 0; d < P; ++d) part_row_base[d + 1] = part_row_base[d] + num_recv_tokens[d];
    // Per local expert of each destination rank, aligned, then offsets.
    for (int32_t d = 0; d < P; ++d) {
        int32_t off = 0;
        for (int32_t l = 0; l < epr; ++l) {
            int64_t cnt = 0;
            for (int32_t s = 0; s < P; ++s) cnt += num_tokens_per_expert[s * E + d * epr + l];
            cnt = ceil_to(cnt, expert_alignment);
            num_recv_tokens_per_expert[d * epr + l] = static_cast<int32_t>(cnt);
            recv_expert_offset[d * epr + l] = off;
            off += static_cast<int32_t>(cnt);
        }
    }
    // Channel prefixes: count is_token_in_rank over each channel's tokens.
    for (int32_t s = 0; s < P; ++s) {
        for (int32_t d = 0; d < P; ++d) {
            int32_t run = 0;
            for (int32_t c = 0; c < C; ++c) {
                int64_t b, e;
                channel_range(T, C, c, &b, &e);
                for (int64_t t = b; t < e; ++t) run += is_token_in_rank[(s * T + t) * P + d];
                channel_prefix_matrix[(static_cast<int64_t>(s) * P + d) * C + c] = run;
            }
        }
    }
    for (int32_t d = 0; d < P; ++d) {
        for (int32_t s = 0; s < P; ++s) {
            for (int32_t c = 0; c < C; ++c) {
                int32_t rank_base = s > 0 ? rank_prefix_matrix[(s - 1) * P + d] : 0;
                int32_t chan_base =
                    c > 0 ? channel_prefix_matrix[(static_cast<int64_t>(s) * P + d) * C + c - 1] : 0;
                recv_channel_prefix_matrix[(static_cast<int64_t>(d) * P + s) * C + c] =
                    rank_base + chan_base;
            }
        }
    }
    // send_head: one counter per destination, tokens in global order.
    for (int32_t d = 0; d < P; ++d) {
        int32_t counter = 0;
        for (int64_t g = 0; g < S; ++g) {
            send_head[g * P + d] = is_token_in_rank[g * P + d] ? counter++ : -1;
        }
    }
}

// Dynamic int8 quantisation of one row [Q]. Writes H int8 and returns scale.
float oracle_quantize_row(int32_t H, const uint16_t* x_row, int8_t* q_row) {
    float amax = 0.0f;
    for (int32_t h = 0; h < H; ++h) {
        float a = std::fabs(bf16_bits_to_float(x_row[h]));
        if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    for (int32_t h = 0; h < H; ++h) {
        int32_t q = 0;
        if (amax != 0.0f) {
            float v = bf16_bits_to_float(x_row[h]) / scale;
            float r = std::nearbyint(v);   // default rounding mode: to nearest, ties to even
            q = static_cast<int32_t>(r);
            if (q > 127) q = 127;
            if (q < -127) q = -127;
        }
        q_row[h] = static_cast<int8_t>(q);
    }
    return scale;
}

// Dispatch [R][H][D][F][Q]. For every token in `tokens` (all tokens in order
// when tokens == NULL) and every destination d (ascending) with
// send_head[g][d] >= 0, writes row part_row_base[d] + send_head[g][d] of the
// arena: payload, scale (quant only), triple; plus the side arrays (each may
// be NULL). Rows that fall outside the partition or the arena are skipped and
// make the return value 3.
int32_t oracle_dispatch(int32_t P, int32_t E, int64_t S, int32_t K, int32_t H, int32_t quant,
                        const uint16_t* x, const int32_t* topk_idx, const float* topk_weights,
                        const int32_t* send_head, const int64_t* part_row_base,
                        uint8_t* arena, int64_t arena_rows,
                        int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                        const int64_t* tokens, int64_t n_tokens) {
    const int32_t epr = E / P;
    const int64_t T = S / P;
    const int64_t stride = oracle_slot_stride(H, quant);
    const int64_t elt = quant ? 1 : 2;
    const int64_t scale_off = ceil_to(static_cast<int64_t>(H) * elt, 32);
    const int64_t triple_off = scale_off + 32;
    int32_t err = 0;
    std::vector<int8_t> q(H);
    const int64_t count = tokens ? n_tokens : S;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t g = tokens ? tokens[i] : i;
        float scale = 0.0f;
        if (quant) scale = oracle_quantize_row(H, x + g * H, q.data());
        for (int32_t d = 0; d < P; ++d) {
            int32_t sh = send_head[g * P + d];
            if (sh < 0) continue;
            if (sh >= part_row_base[d + 1] - part_row_base[d]) { err = 3; continue; }
            int64_t row = part_row_base[d] + sh;
            if (row >= arena_rows) { err = 3; continue; }
            uint8_t* slot = arena + row * stride;
            if (quant) {
                std::memcpy(slot, q.data(), H);
                std::memcpy(slot + scale_off, &scale, 4);
            } else {
                std::memcpy(slot, x + g * H, static_cast<size_t>(H) * 2);
            }
            int32_t kmin = -1;
            for (int32_t k = 0; k < K; ++k) {
                if (slot_on_rank(topk_idx[g * K + k], E, epr, d)) { kmin = k; break; }
            }
            int32_t triple[3] = {static_cast<int32_t>(g / T), static_cast<int32_t>(g % T), kmin};
            std::memcpy(slot + triple_off, triple, 12);
            if (recv_src_idx) recv_src_idx[row] = static_cast<int32_t>(g % T);
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = topk_idx[g * K + k];
                bool on = slot_on_rank(e, E, epr, d);
                if (recv_topk_idx) recv_topk_idx[row * K + k] = on ? e % epr : -1;
                if (recv_topk_weights) recv_topk_weights[row * K + k] = on ? topk_weights[g * K + k] : 0.0f;
            }
        }
    }
    return err;
}

// Combine [R][C]. For every token in `tokens` (all when NULL):
//   out[g] = bf16_rne( sum over d ascending with send_head[g][d] >= 0 of
//                      c_{g,d} * f32(y[part_row_base[d] + send_head[g][d]]) )
// accumulated in binary32, each product and sum rounded on its own.
// y rows are y_row_stride bytes apart. Out-of-range rows are skipped and make
// the return value 3.
int32_t oracle_combine(int32_t P, int32_t E, int64_t S, int32_t K, int32_t H,
                       const uint8_t* y, int64_t y_row_stride, const int64_t* part_row_base,
                       int64_t arena_rows, const int32_t* send_head, const int32_t* topk_idx,
                       const float* topk_weights, uint16_t* out,
                       const int64_t* tokens, int64_t n_tokens) {
    const int32_t epr = E / P;
    int32_t err = 0;
    std::vector<float> acc(H);
    const int64_t count = tokens ? n_tokens : S;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t g = tokens ? tokens[i] : i;
        std::fill(acc.begin(), acc.end(), 0.0f);
        for (int32_t d = 0; d < P; ++d) {
            int32_t sh = send_head[g * P + d];
            if (sh < 0) continue;
            if (sh >= part_row_base[d + 1] - part_row_base[d]) { err = 3; continue; }
            int64_t row = part_row_base[d] + sh;
            if (row >= arena_rows) { err = 3; continue; }
            float c;
            if (topk_weights) {
                c = 0.0f;
                for (int32_t k = 0; k < K; ++k) {
                    if (slot_on_rank(topk_idx[g * K + k], E, epr, d)) c = c + topk_weights[g * K + k];
                }
            } else {
                c = 1.0f;
            }
            const uint16_t* yrow = reinterpret_cast<const uint16_t*>(y + row * y_row_stride);
            for (int32_t h = 0; h < H; ++h) {
                float prod = c * bf16_bits_to_float(yrow[h]);
                acc[h] = acc[h] + prod;
            }
        }
        for (int32_t h = 0; h < H; ++h) out[g * H + h] = float_to_bf16_bits_rne(acc[h]);
    }
    return err;
}

// ---- Expert-major receive layout --------------------------------------------
// "HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 3.6 (InputToShare): each
// (token, k) slot is copied to hOutGMAlignSize * (dstExpertOffset +
// curExpertCnt) of its expert's rank, the triple carrying that slot's k; and
// section 7.8 (ReadBufferAndWeightedSum): the owner sums the K returned rows,
// weight by weight, in k order. Inside rank d, expert l's rows start at
// recv_expert_offset[d][l] (its aligned count's exclusive scan, "internode.cu"
// section 1) and hold the expert's slots in (token, k) order.

// slot_row[g][k] = recv_expert_offset[d][l] + (slots with the same expert that
// come before (g, k) in (token, k) order), or -1 for a masked / invalid slot.
// expert_part_base = exclusive scan over ranks of sum_l num_recv_tokens_per_expert[d][l].
void oracle_notify_expert(int32_t P, int32_t E, int64_t S, int32_t K, const int32_t* topk_idx,
                          const int32_t* num_recv_tokens_per_expert, const int32_t* recv_expert_offset,
                          int32_t* slot_row, int64_t* expert_part_base) {
    const int32_t epr = E / P;
    std::vector<int32_t> counter(E, 0);
    for (int64_t g = 0; g < S; ++g) {
        for (int32_t k = 0; k < K; ++k) {
            const int32_t e = topk_idx[g * K + k];
            if (e < 0 || e >= E) {
                slot_row[g * K + k] = -1;
                continue;
            }
            slot_row[g * K + k] = recv_expert_offset[e] + counter[e];
            counter[e] += 1;
        }
    }
    expert_part_base[0] = 0;
    for (int32_t d = 0; d < P; ++d) {
        int64_t total = 0;
        for (int32_t l = 0; l < epr; ++l) total += num_recv_tokens_per_expert[d * epr + l];
        expert_part_base[d + 1] = expert_part_base[d] + total;
    }
}

// One slot per valid (g, k): row expert_part_base[d] + slot_row[g][k] receives
// the payload (as in oracle_dispatch), the triple (g / T, g % T, k),
// recv_src_idx = g % T and recv_weight = topk_weights[g][k] (side arrays may
// be NULL). Rows outside the partition or the arena are skipped: return 3.
int32_t oracle_dispatch_expert(int32_t P, int32_t E, int64_t S, int32_t K, int32_t H, int32_t quant,
                               const uint16_t* x, const int32_t* topk_idx, const float* topk_weights,
                               const int32_t* slot_row, const int64_t* expert_part_base,
                               uint8_t* arena, int64_t arena_rows, int32_t* recv_src_idx,
                               float* recv_weight, const int64_t* tokens, int64_t n_tokens) {
    const int32_t epr = E / P;
    const int64_t T = S / P;
    const int64_t stride = oracle_slot_stride(H, quant);
    const int64_t elt = quant ? 1 : 2;
    const int64_t scale_off = ceil_to(static_cast<int64_t>(H) * elt, 32);
    const int64_t triple_off = scale_off + 32;
    int32_t err = 0;
    std::vector<int8_t> q(H);
    const int64_t count = tokens ? n_tokens : S;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t g = tokens ? tokens[i] : i;
        float scale = 0.0f;
        if (quant) scale = oracle_quantize_row(H, x + g * H, q.data());
        for (int32_t k = 0; k < K; ++k) {
            const int32_t e = topk_idx[g * K + k];
            const int32_t sr = slot_row[g * K + k];
            if (e < 0 || e >= E || sr < 0) continue;
            const int32_t d = e / epr;
            if (sr >= expert_part_base[d + 1] - expert_part_base[d]) { err = 3; continue; }
            const int64_t row = expert_part_base[d] + sr;
            if (row >= arena_rows) { err = 3; continue; }
            uint8_t* slot = arena + row * stride;
            if (quant) {
                std::memcpy(slot, q.data(), H);
                std::memcpy(slot + scale_off, &scale, 4);
            } else {
                std::memcpy(slot, x + g * H, static_cast<size_t>(H) * 2);
            }
            const int32_t triple[3] = {static_cast<int32_t>(g / T), static_cast<int32_t>(g % T), k};
            std::memcpy(slot + triple_off, triple, 12);
            if (recv_src_idx) recv_src_idx[row] = static_cast<int32_t>(g % T);
            if (recv_weight) recv_weight[row] = topk_weights ? topk_weights[g * K + k] : 1.0f;
        }
    }
    return err;
}

// out[g] = bf16_rne( sum over k ascending with a valid slot of
//                    w[g][k] * f32(y[expert_part_base[d] + slot_row[g][k]]) ),
// binary32 accumulator from +0, product and sum rounded separately; NULL
// weights mean w = 1.
int32_t oracle_combine_expert(int32_t P, int32_t E, int64_t S, int32_t K, int32_t H,
                              const uint8_t* y, int64_t y_row_stride, const int64_t* expert_part_base,
                              int64_t arena_rows, const int32_t* slot_row, const int32_t* topk_idx,
                              const float* topk_weights, uint16_t* out, const int64_t* tokens,
                              int64_t n_tokens) {
    const int32_t epr = E / P;
    int32_t err = 0;
    std::vector<float> acc(H);
    const int64_t count = tokens ? n_tokens : S;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t g = tokens ? tokens[i] : i;
        std::fill(acc.begin(), acc.end(), 0.0f);
        for (int32_t k = 0; k < K; ++k) {
            const int32_t e = topk_idx[g * K + k];
            const int32_t sr = slot_row[g * K + k];
            if (e < 0 || e >= E || sr < 0) continue;
            const int32_t d = e / epr;
            if (sr >= expert_part_base[d + 1] - expert_part_base[d]) { err = 3; continue; }
            const int64_t row = expert_part_base[d] + sr;
            if (row >= arena_rows) { err = 3; continue; }
            const float w = topk_weights ? topk_weights[g * K + k] : 1.0f;
            const uint16_t* yrow = reinterpret_cast<const uint16_t*>(y + row * y_row_stride);
            for (int32_t h = 0; h < H; ++h) {
                float prod = w * bf16_bits_to_float(yrow[h]);
                acc[h] = acc[h] + prod;
            }
        }
        for (int32_t h = 0; h < H; ++h) out[g * H + h] = float_to_bf16_bits_rne(acc[h]);
    }
    return err;
}

// Fixed-length receive partitions ("Ascend DeepEP MoE Dispatch Optimization",
// section "输出长度有动态和固定两种模式": with a fixed output length the rows
// past the received count are padding -- x, scales and weights 0, topk_idx
// -1). For every rank d the rows part_row_base[d] + num_recv_tokens[d] up to
// part_row_base[d+1] (and below arena_rows) get: payload 0; the scale block 0
// (int8); the triple (-1, -1, -1); recv_src_idx -1; recv_topk_idx -1;
// recv_topk_weights 0.
void oracle_pad_partitions(int32_t P, int32_t K, int32_t H, int32_t quant,
                           const int32_t* num_recv_tokens, const int64_t* part_row_base,
                           uint8_t* arena, int64_t arena_rows, int32_t* recv_src_idx,
                           int32_t* recv_topk_idx, float* recv_topk_weights) {
    const int64_t stride = oracle_slot_stride(H, quant);
    const int64_t elt = quant ? 1 : 2;
    const int64_t scale_off = ceil_to(static_cast<int64_t>(H) * elt, 32);
    const int64_t triple_off = scale_off + 32;
    for (int32_t d = 0; d < P; ++d) {
        for (int64_t r = part_row_base[d] + num_recv_tokens[d]; r < part_row_base[d + 1]; ++r) {
            if (r < 0 || r >= arena_rows) continue;
            uint8_t* slot = arena + r * stride;
            std::memset(slot, 0, static_cast<size_t>(H) * elt);
            if (quant) std::memset(slot + scale_off, 0, 32);
            const int32_t triple[3] = {-1, -1, -1};
            std::memcpy(slot + triple_off, triple, 12);
            if (recv_src_idx) recv_src_idx[r] = -1;
            for (int32_t k = 0; k < K; ++k) {
                if (recv_topk_idx) recv_topk_idx[r * K + k] = -1;
                if (recv_topk_weights) recv_topk_weights[r * K + k] = 0.0f;
            }
        }
    }
}

// Exposed for the pin tests of the conversion helpers.
void oracle_bf16_round(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16_bits_rne(in[i]);
}

}  // extern "C"
