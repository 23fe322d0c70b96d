/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for the token
 * layout -> dispatch -> TransferCmd descriptors -> combine of one
 * expert-parallel (EP) layer whose R ranks are partitions of one buffer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this.  It shares no code, header, table or helper
 * with the CUDA path; it is written directly from the definitions below, by
 * plain loops, in the order the definitions state them.
 *
 * Sources (web articles on MoE expert-parallel communication):
 *  [UCCL-EP]  "UCCL-EP: GPU-side FIFO queues and CPU proxy threads"
 *             (peacm.com/news/835744).  s1: EP needs fine-grained token-level
 *             communication; s2.2: the FIFO ring of TransferCmd records;
 *             s2.3: TransferCmd{dst_rank, src_offset, dst_offset, size};
 *             s4.1: small tokens (< 7 KB) are packed into one message;
 *             s4.2: 8 independent FIFOs per GPU; s5.2: tuning table;
 *             s6: EP32 dispatch / combine.
 *  [GIN]      "NCCL GIN: device-initiated GPU networking"
 *             (bjdmk.com.cn/news/2086017).  s2.2.1: windows addressed by
 *             byte offset.
 *  [NOTES]    "GPU communication mechanisms and optimisation techniques"
 *             (blog.zhenwei.site), table "software communication stack":
 *             layout/rank mismatch is a named failure class of EP dispatch.
 *
 * Readings taken where the articles are silent (each one is also listed with
 * the design notes):
 *  - expert e lives on rank e / (E/R) (contiguous blocks of experts);
 *  - one receive row per (token, destination rank), however many of the
 *    token's experts live on that rank;
 *  - receive rows of rank d are ordered by global token index (tokens are
 *    numbered source-rank-major, so this is source rank, then token);
 *  - topk_idx == -1 means "no pick"; any other value outside [0, E) is an
 *    invalid argument;
 *  - a message carries up to G consecutive rows of one (source, destination)
 *    pair; src_offset is a byte offset into the logical send buffer whose rows
 *    are ordered (source, destination, row); dst_offset is a byte offset into
 *    the destination rank's receive window; the channel is dst_rank mod C;
 *  - combine: acc = +0.0f, then acc = fmaf(w[t,k], row_k[h], acc) for
 *    k = 0..K-1, where row_k is the receive row of (t, rank of pick k); the
 *    result is rounded to bf16 to nearest, ties to even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_TOPK 1
#define ORACLE_BAD_ARG 2

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 bits -> float: bf16 is the upper half of an IEEE binary32. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float -> bf16 bits, round to nearest, ties to even.  Adding 0x7FFF plus
 * the lowest kept bit to the binary32 pattern and truncating rounds the
 * dropped 16 bits to nearest with ties going to the even kept value; a carry
 * out of the mantissa correctly bumps the exponent.  NaN maps to 0x7FC0 with
 * its sign (the inputs of this layer are finite, so NaN is never compared). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + keep_lsb;
    return (uint16_t)(u >> 16);
}

float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }

/* fp32 fused multiply-add, rounded once (C99 fmaf). */
float oracle_fmaf(float a, float b, float c) { return fmaf(a, b, c); }

/* -------------------------------------------------------------- layout -- */

/*
 * Token layout of one EP layer (the counts, membership and exclusive-scan
 * offsets the EP dispatch needs; [UCCL-EP] s1 token-level routing).
 *
 *   num_tokens_per_expert[s][e] = #{(t, k) : t on rank s, topk_idx[t][k] = e}
 *   is_token_in_rank[t][d]      = 1 if some pick k of t has rank(topk_idx[t][k]) = d
 *   num_tokens_per_rank[s][d]   = sum over t on rank s of is_token_in_rank[t][d]
 *   token_slot[t][d]            = #{t' < t : is_token_in_rank[t'][d]}, or -1
 *   recv_count[d]               = sum_s num_tokens_per_rank[s][d]
 *   recv_base[d]                = sum_{d' < d} recv_count[d']
 *   recv_off[s][d]              = sum_{s' < s} num_tokens_per_rank[s'][d]
 *   send_off[s][d]              = sum of num_tokens_per_rank over all (s', d')
 *                                 before (s, d) in row-major order
 *   msg_count[s][d]             = ceil(num_tokens_per_rank[s][d] / G)
 *   expert_off[e]               = sum_{e' < e} sum_s num_tokens_per_expert[s][e']
 *   n_recv                      = sum_d recv_count[d]
 *
 * All outputs are overwritten.  Returns ORACLE_BAD_TOPK (and stops) when a
 * pick is outside [-1, E).
 */
int oracle_layout(int R, int Tpr, int E, int K, int G, const int32_t *topk_idx,
                  int32_t *num_tokens_per_expert, int32_t *num_tokens_per_rank,
                  uint8_t *is_token_in_rank, int32_t *token_slot,
                  int32_t *recv_off, int32_t *send_off, int32_t *msg_count,
                  int32_t *recv_count, int32_t *recv_base, int32_t *expert_off,
                  int64_t *n_recv) {
    if (R <= 0 || Tpr < 0 || E <= 0 || K <= 0 || G <= 0 || E % R != 0)
        return ORACLE_BAD_ARG;
    const int64_t T = (int64_t)R * Tpr;
    const int Er = E / R;

    memset(num_tokens_per_expert, 0, sizeof(int32_t) * (size_t)R * E);
    memset(is_token_in_rank, 0, (size_t)T * R);

    /* 1. per-expert histogram and rank membership, by direct loops */
    for (int64_t t = 0; t < T; ++t) {
        int s = (int)(t / Tpr);
        for (int k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) return ORACLE_BAD_TOPK;
            num_tokens_per_expert[(int64_t)s * E + e] += 1;
            is_token_in_rank[t * R + e / Er] = 1;
        }
    }

    /* 2. per-(source, destination) counts */
    for (int s = 0; s < R; ++s)
        for (int d = 0; d < R; ++d) {
            int32_t c = 0;
            for (int64_t t = (int64_t)s * Tpr; t < (int64_t)(s + 1) * Tpr; ++t)
                c += is_token_in_rank[t * R + d];
            num_tokens_per_rank[s * R + d] = c;
        }

    /* 3. receive slot of each (token, destination): a running counter down
     *    each destination column, in increasing token order */
    for (int d = 0; d < R; ++d) {
        int32_t running = 0;
        for (int64_t t = 0; t < T; ++t) {
            if (is_token_in_rank[t * R + d]) {
                token_slot[t * R + d] = running;
                running += 1;
            } else {
                token_slot[t * R + d] = -1;
            }
        }
    }

    /* 4. the small scans */
    for (int d = 0; d < R; ++d) {
        int32_t c = 0;
        for (int s = 0; s < R; ++s) c += num_tokens_per_rank[s * R + d];
        recv_count[d] = c;
    }
    {
        int32_t acc = 0;
        for (int d = 0; d < R; ++d) {
            recv_base[d] = acc;
            acc += recv_count[d];
        }
    }
    for (int d = 0; d < R; ++d) {
        int32_t acc = 0;
        for (int s = 0; s < R; ++s) {
            recv_off[s * R + d] = acc;
            acc += num_tokens_per_rank[s * R + d];
        }
    }
    {
        int32_t acc = 0;
        for (int s = 0; s < R; ++s)
            for (int d = 0; d < R; ++d) {
                send_off[s * R + d] = acc;
                acc += num_tokens_per_rank[s * R + d];
            }
    }
    for (int i = 0; i < R * R; ++i)
        msg_count[i] = (num_tokens_per_rank[i] + G - 1) / G;
    {
        int32_t acc = 0;
        for (int e = 0; e < E; ++e) {
            expert_off[e] = acc;
            for (int s = 0; s < R; ++s) acc += num_tokens_per_expert[(int64_t)s * E + e];
        }
    }
    {
        int64_t n = 0;
        for (int d = 0; d < R; ++d) n += recv_count[d];
        *n_recv = n;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------ dispatch -- */

/*
 * Dispatch ([UCCL-EP] s6 "Dispatch"): for every token t in [t_begin, t_end)
 * and every destination d with token_slot[t][d] >= 0, copy the row_bytes of
 * x[t] to recv row recv_base[d] + token_slot[t][d].  One copy per
 * (token, destination rank).  Rows are opaque bytes.
 */
void oracle_dispatch(int R, int64_t t_begin, int64_t t_end, int64_t row_bytes,
                     const int32_t *token_slot, const int32_t *recv_base,
                     const uint8_t *x, uint8_t *recv) {
    for (int64_t t = t_begin; t < t_end; ++t)
        for (int d = 0; d < R; ++d) {
            int32_t slot = token_slot[t * R + d];
            if (slot < 0) continue;
            int64_t row = (int64_t)recv_base[d] + slot;
            memcpy(recv + row * row_bytes, x + t * row_bytes, (size_t)row_bytes);
        }
}

/* --------------------------------------------------------- descriptors -- */

/* One ring record ([UCCL-EP] s2.3 TransferCmd fields), 32 bytes. */
typedef struct {
    uint32_t dst_rank;
    uint32_t size;
    uint64_t src_offset;
    uint64_t dst_offset;
    uint32_t type; /* 0 = WRITE */
    uint32_t reserved;
} oracle_cmd;

/* Number of messages each channel receives: channel c carries every message
 * whose destination rank d has d mod C == c ([UCCL-EP] s4.2, 8 FIFOs). */
void oracle_channel_counts(int R, int C, const int32_t *msg_count, int64_t *per_channel) {
    for (int c = 0; c < C; ++c) per_channel[c] = 0;
    for (int s = 0; s < R; ++s)
        for (int d = 0; d < R; ++d) per_channel[d % C] += msg_count[s * R + d];
}

/*
 * The TransferCmd list in canonical order: channel-major; within a channel,
 * source s ascending, then destination d ascending, then message g ascending.
 * Message g of pair (s, d) carries rows j in [g*G, min(g*G + G, cnt)) where
 * cnt = num_tokens_per_rank[s][d]; its payload is n = min(G, cnt - g*G) rows:
 *   size       = n * row_bytes
 *   src_offset = (send_off[s][d] + g*G) * row_bytes    (logical send buffer)
 *   dst_offset = (recv_off[s][d] + g*G) * row_bytes    (window of rank d)
 * out must hold sum_c per_channel[c] records; channel c starts at
 * sum_{c' < c} per_channel[c'].
 */
void oracle_descriptors(int R, int C, int G, int64_t row_bytes,
                        const int32_t *num_tokens_per_rank, const int32_t *recv_off,
                        const int32_t *send_off, oracle_cmd *out) {
    int64_t *fill = (int64_t *)calloc((size_t)C, sizeof(int64_t));
    int64_t *start = (int64_t *)calloc((size_t)C, sizeof(int64_t));
    int64_t *per = (int64_t *)calloc((size_t)C, sizeof(int64_t));
    for (int s = 0; s < R; ++s)
        for (int d = 0; d < R; ++d)
            per[d % C] += (num_tokens_per_rank[s * R + d] + G - 1) / G;
    for (int c = 1; c < C; ++c) start[c] = start[c - 1] + per[c - 1];
    for (int c = 0; c < C; ++c)
        for (int s = 0; s < R; ++s)
            for (int d = 0; d < R; ++d) {
                if (d % C != c) continue;
                int32_t cnt = num_tokens_per_rank[s * R + d];
                for (int32_t j0 = 0; j0 < cnt; j0 += G) {
                    int32_t n = cnt - j0 < G ? cnt - j0 : G;
                    oracle_cmd *m = &out[start[c] + fill[c]];
                    m->dst_rank = (uint32_t)d;
                    m->size = (uint32_t)((int64_t)n * row_bytes);
                    m->src_offset = (uint64_t)(((int64_t)send_off[s * R + d] + j0) * row_bytes);
                    m->dst_offset = (uint64_t)(((int64_t)recv_off[s * R + d] + j0) * row_bytes);
                    m->type = 0;
                    m->reserved = 0;
                    fill[c] += 1;
                }
            }
    free(fill);
    free(start);
    free(per);
}

/* ------------------------------------------------------------- combine -- */

/*
 * Combine ([UCCL-EP] s6 "Combine"): for every token t in [t_begin, t_end),
 *   out[t][h] = bf16_rne( fmaf-chain over k = 0..K-1 of
 *                         topk_weights[t][k] * expert_out[row(t, k)][h] )
 * with the chain starting from +0.0f, row(t, k) = recv_base[d] +
 * token_slot[t][d], d = topk_idx[t][k] / Er.  Picks equal to -1 add nothing.
 * Returns ORACLE_BAD_ARG if a row falls outside [0, n_rows).
 */
int oracle_combine(int R, int Er, int K, int64_t H, int64_t t_begin, int64_t t_end,
                   const int32_t *topk_idx, const float *topk_weights,
                   const int32_t *token_slot, const int32_t *recv_base,
                   const uint16_t *expert_out, int64_t n_rows, uint16_t *out) {
    float *acc = (float *)malloc(sizeof(float) * (size_t)H);
    if (!acc) return ORACLE_BAD_ARG;
    for (int64_t t = t_begin; t < t_end; ++t) {
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e == -1) continue;
            int d = e / Er;
            if (d < 0 || d >= R) { free(acc); return ORACLE_BAD_ARG; }
            int32_t slot = token_slot[t * R + d];
            int64_t row = (int64_t)recv_base[d] + slot;
            if (slot < 0 || row < 0 || row >= n_rows) { free(acc); return ORACLE_BAD_ARG; }
            float w = topk_weights[t * K + k];
            const uint16_t *src = expert_out + row * H;
            for (int64_t h = 0; h < H; ++h) acc[h] = fmaf(w, bf16_to_f32(src[h]), acc[h]);
        }
        for (int64_t h = 0; h < H; ++h) out[(t - t_begin) * H + h] = oracle_f32_to_bf16(acc[h]);
    }
    free(acc);
    return ORACLE_OK;
}

/* ------------------------------------------------------- expert layout -- */

/*
 * Expert-major receive metadata: what a rank needs after dispatch to run its
 * local experts on the rows it received ([UCCL-EP] s1: each token goes to the
 * experts of its top-k picks; the grouped expert step consumes the received
 * rows per expert).
 *
 * For every receive row n = recv_base[d] + token_slot[t][d]:
 *   recv_src_token[n]       = t
 *   recv_topk_idx[n][k]     = topk_idx[t][k] - d*Er  if pick k lives on rank d,
 *                             else -1
 *   recv_topk_weights[n][k] = topk_weights[t][k]     if pick k lives on rank d,
 *                             else 0.0f
 * and, taking the picks (t, k) in increasing t, then k:
 *   expert_rows[expert_off[e] + j] = receive row of the j-th pick of expert e
 *                                    (row of (t, rank of e))
 *   expert_count[e]                = number of picks of expert e
 * expert_rows therefore lists, per expert, the rows it must process in
 * increasing receive-row order.  A token naming one expert twice has no
 * well-defined position and is rejected (ORACLE_BAD_TOPK), as is a pick
 * outside [-1, E).  recv_* must hold n_recv rows; expert_rows must hold one
 * entry per pick that is not -1.
 */
int oracle_expert_layout(int R, int Tpr, int E, int K, const int32_t *topk_idx,
                         const float *topk_weights, const int32_t *token_slot,
                         const int32_t *recv_base, const int32_t *expert_off, int64_t n_recv,
                         int32_t *recv_topk_idx, float *recv_topk_weights,
                         int32_t *recv_src_token, int32_t *expert_rows, int32_t *expert_count) {
    if (R <= 0 || Tpr < 0 || E <= 0 || K <= 0 || E % R != 0) return ORACLE_BAD_ARG;
    const int64_t T = (int64_t)R * Tpr;
    const int Er = E / R;

    /* picks must be -1 or an expert, and distinct within a token */
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) return ORACLE_BAD_TOPK;
            for (int k2 = 0; k2 < k; ++k2)
                if (topk_idx[t * K + k2] == e) return ORACLE_BAD_TOPK;
        }

    /* 1. per receive row: source token, local picks and their weights */
    for (int64_t t = 0; t < T; ++t)
        for (int d = 0; d < R; ++d) {
            int32_t slot = token_slot[t * R + d];
            if (slot < 0) continue;
            int64_t n = (int64_t)recv_base[d] + slot;
            if (n < 0 || n >= n_recv) return ORACLE_BAD_ARG;
            recv_src_token[n] = (int32_t)t;
            for (int k = 0; k < K; ++k) {
                int32_t e = topk_idx[t * K + k];
                if (e >= 0 && e / Er == d) {
                    recv_topk_idx[n * K + k] = e - d * Er;
                    recv_topk_weights[n * K + k] = topk_weights[t * K + k];
                } else {
                    recv_topk_idx[n * K + k] = -1;
                    recv_topk_weights[n * K + k] = 0.0f;
                }
            }
        }

    /* 2. per expert: its picks' receive rows, in pick order */
    for (int e = 0; e < E; ++e) expert_count[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e < 0) continue;
            int d = e / Er;
            int64_t row = (int64_t)recv_base[d] + token_slot[t * R + d];
            expert_rows[(int64_t)expert_off[e] + expert_count[e]] = (int32_t)row;
            expert_count[e] += 1;
        }
    return ORACLE_OK;
}

/* ------------------------------------------------------------- signals -- */

/*
 * Arrival signals ([GIN] s2.2.2 completion notification: a put may carry a
 * signal increment that the destination reads as remote completion; s2.1.2
 * put with SignalInc, then waitSignal on an expected value).  With one signal
 * per destination rank, incremented once per message that lands there, a
 * dispatch leaves
 *   signal[d] = number of messages of that dispatch with dst_rank d
 *             = sum over s of msg_count[s][d].
 */
void oracle_signal_counts(int R, const int32_t *msg_count, uint64_t *signal) {
    for (int d = 0; d < R; ++d) {
        uint64_t n = 0;
        for (int s = 0; s < R; ++s) n += (uint64_t)msg_count[s * R + d];
        signal[d] = n;
    }
}
