// ep_expert.cu -- expert-major receive metadata of one EP layer (sm_103a).
//
// What it computes (UCCL-EP article s1: each token goes to the experts of its
// top-k picks; the receiving rank runs those experts on the rows it got):
//   per receive row n = recv_base[d] + token_slot[t][d]: the source token t,
//   and the token's picks that live on rank d as local expert ids with their
//   weights (-1 / 0 elsewhere);
//   per expert e: the receive rows of its picks in token order, placed at
//   expert_off[e] + j, and the count of its picks.
//
// How: one CTA per tile of 256 tokens (128 when E > 2048; one token per
// thread), tiles handed out in launch order by a ticket counter, so a tile's
// predecessors are already running.  Per tile:
//   1. each thread holds its token's K picks and weights in registers,
//      checks them (range, no expert named twice), and sets its bit in the
//      tile's bitmask of each picked expert (shared memory, E x TILE/32 words);
//   2. per expert column: the tile's count is the popcount of its mask;
//      decoupled look-back (Merrill & Garland, "Single-pass Parallel Prefix
//      Scan with Decoupled Look-back", 2016) over the preceding tiles gives
//      the picks of that expert in earlier tokens.  All columns' aggregates
//      are published before any look-back starts.  A descriptor is one 64-bit
//      word {epoch:30 | flag:2 | value:32}; the epoch comes from the ticket,
//      so nothing is reset between calls (CUDA-graph safe);
//   3. the metadata of each receive row the token owns (one row per rank it
//      reaches; K-wide vector stores where K % 4 == 0) -- after the look-back,
//      so successors never wait on these stores -- and each pick's position =
//      expert_off[e] + earlier tiles + popcount of the mask bits of earlier
//      tokens in this tile; expert_rows gets the pick's receive row there.
// Reads T*K*8 (picks, weights) plus each pick's token_slot entry; writes
// N*(8K + 4) + M*4 + E*4 bytes.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kXTileSmall = 128;          // tokens per tile when E is large
constexpr int kXTileLarge = 256;          // tokens per tile when E <= kXLargeMaxE
constexpr int kXLargeMaxE = 2048;
constexpr int kPickBatch = 4;             // picks whose loads are in flight together

struct ExpertParams {
    const int32_t *topk_idx;
    const float *topk_weights;
    const int32_t *token_slot;
    const int32_t *recv_base;
    const int32_t *expert_off;
    ep_expert_layout_out out;
    DevState dev;
    int64_t T, recv_rows, rows_cap;
    uint64_t timeout_ns;
    int R, E, K, Er;
    int tiles;
    int vec4;              // K % 4 == 0 and the row outputs are 16-byte aligned
    int vec8;              // K % 8 == 0 and the row outputs are 32-byte aligned
};

// One 32-byte store (st.global.v8.b32); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// K <= 8: four CTAs per SM (at most 64 registers a thread at 256 threads), so
// that a 512-tile layer runs in one wave.
template <int KMAX, int TILE>
__global__ void __launch_bounds__(TILE, KMAX <= 8 ? 4 : 1) expert_layout_kernel(const ExpertParams p) {
    constexpr int kXWords = TILE / 32;   // mask words per expert (one per warp)
    extern __shared__ __align__(16) uint32_t s_mask[];    // [E][kXWords], then s_excl[E]
    __shared__ unsigned long long s_ticket;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = p.R, E = p.E, K = p.K, Er = p.Er;
    int *s_excl = reinterpret_cast<int *>(s_mask + static_cast<size_t>(E) * kXWords);

    if (tid == 0) s_ticket = atomicAdd(p.dev.xticket, 1ull);
    for (int i = tid; i < E * kXWords; i += TILE) s_mask[i] = 0u;
    __syncthreads();
    const unsigned long long ticket = s_ticket;
    const int tile = static_cast<int>(ticket % static_cast<unsigned long long>(p.tiles));
    const uint32_t epoch = static_cast<uint32_t>((ticket / p.tiles) % ((1u << 30) - 1u)) + 1u;
    const int64_t t = static_cast<int64_t>(tile) * TILE + tid;
    const bool valid = t < p.T;

    // 1. picks and weights in registers; -1 marks "no pick" and bad picks
    int pk[KMAX];
    float wk[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        pk[k] = -1;
        wk[k] = 0.0f;
        if (valid && k < K) {
            int e = __ldg(p.topk_idx + t * K + k);
            if (e < -1 || e >= E) {
                set_error(p.dev.err, EP_ERR_INVALID_ARG);
                e = -1;
            }
#pragma unroll
            for (int k2 = 0; k2 < k; ++k2)
                if (e >= 0 && pk[k2] == e) {
                    set_error(p.dev.err, EP_ERR_INVALID_ARG);
                    e = -1;
                }
            pk[k] = e;
            wk[k] = __ldg(p.topk_weights + t * K + k);
        }
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
        if (pk[k] >= 0) atomicOr(&s_mask[pk[k] * kXWords + warp], 1u << lane);

    __syncthreads();

    // 2. per expert column: publish every aggregate, then look back
    unsigned long long *desc = p.dev.xdesc + static_cast<int64_t>(tile) * E;
    for (int e = tid; e < E; e += TILE) {
        const uint32_t *m = s_mask + e * kXWords;
        int agg = 0;
#pragma unroll
        for (int w = 0; w < kXWords; ++w) agg += __popc(m[w]);
        s_excl[e] = agg;
        st_relaxed(desc + e, look_desc(epoch, tile == 0 ? kLookPrefix : kLookAggregate,
                                         static_cast<uint32_t>(agg)));
    }
    const uint64_t t_start = globaltimer_ns();
    for (int e = tid; e < E; e += TILE) {
        const int agg = s_excl[e];
        int excl = 0;
        if (tile > 0) {
            excl = lookback_excl(p.dev.xdesc, E, e, tile, epoch, t_start, p.timeout_ns, p.dev.err);
            st_relaxed(desc + e, look_desc(epoch, kLookPrefix, static_cast<uint32_t>(excl + agg)));
        }
        s_excl[e] = excl;
        if (tile == p.tiles - 1) p.out.expert_count[e] = excl + agg;
    }
    __syncthreads();

    // 3. per pick, in batches of kPickBatch: first every load the batch
    //    needs (the receive row of the pick's rank, its expert's offset) --
    //    one round trip -- then the stores.
    //    a. per-row metadata: one receive row per rank the token reaches,
    //       written at its first pick on that rank (after the look-back, so
    //       successors never wait on these stores);
    //    b. the pick's place in its expert's segment: expert_off[e] + earlier
    //       tiles + mask bits of earlier tokens in this tile.
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int k0 = 0; k0 < KMAX; k0 += kPickBatch) {
        int64_t row[kPickBatch];
        int eoff[kPickBatch];
#pragma unroll
        for (int b = 0; b < kPickBatch; ++b) {
            const int e = pk[k0 + b];
            row[b] = -1;
            eoff[b] = 0;
            if (e >= 0) {
                const int d = e / Er;
                const int slot = __ldg(p.token_slot + t * R + d);
                row[b] = slot >= 0 ? static_cast<int64_t>(__ldg(p.recv_base + d)) + slot : -1;
                eoff[b] = __ldg(p.expert_off + e);
            }
        }
#pragma unroll
        for (int b = 0; b < kPickBatch; ++b) {
            const int k = k0 + b;
            const int e = pk[k];
            if (e < 0) continue;
            const int d = e / Er;
            const int64_t n = row[b];
            if (n < 0) {
                set_error(p.dev.err, EP_ERR_INVALID_ARG);    // layout of another routing
                continue;
            }
            bool first = true;
#pragma unroll
            for (int k2 = 0; k2 < k; ++k2)
                if (pk[k2] >= 0 && pk[k2] / Er == d) first = false;
            if (first) {
                if (n >= p.recv_rows) {
                    set_error(p.dev.err, EP_ERR_CAPACITY);
                } else {
                    p.out.recv_src_token[n] = static_cast<int32_t>(t);
                    const int lo = d * Er;
                    if (p.vec8) {
                        // whole 32-byte sectors: one store per eight picks
                        int32_t *ri = p.out.recv_topk_idx + n * K;
                        float *rw = p.out.recv_topk_weights + n * K;
#pragma unroll
                        for (int k8 = 0; k8 < KMAX; k8 += 8) {
                            if (k8 >= K) break;
                            uint32_t v[8], u[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int ej = pk[k8 + j];
                                const bool on = ej >= 0 && ej / Er == d;
                                v[j] = static_cast<uint32_t>(on ? ej - lo : -1);
                                u[j] = __float_as_uint(on ? wk[k8 + j] : 0.0f);
                            }
                            st_global_v8(ri + k8, v);
                            st_global_v8(rw + k8, u);
                        }
                    } else if (p.vec4) {
                        int4 *ri = reinterpret_cast<int4 *>(p.out.recv_topk_idx + n * K);
                        float4 *rw = reinterpret_cast<float4 *>(p.out.recv_topk_weights + n * K);
#pragma unroll
                        for (int k4 = 0; k4 < KMAX; k4 += 4) {
                            if (k4 >= K) break;
                            int v[4];
                            float u[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int ej = pk[k4 + j];
                                const bool on = ej >= 0 && ej / Er == d;
                                v[j] = on ? ej - lo : -1;
                                u[j] = on ? wk[k4 + j] : 0.0f;
                            }
                            ri[k4 / 4] = make_int4(v[0], v[1], v[2], v[3]);
                            rw[k4 / 4] = make_float4(u[0], u[1], u[2], u[3]);
                        }
                    } else {
#pragma unroll
                        for (int k2 = 0; k2 < KMAX; ++k2) {
                            if (k2 >= K) break;
                            const int ej = pk[k2];
                            const bool on = ej >= 0 && ej / Er == d;
                            p.out.recv_topk_idx[n * K + k2] = on ? ej - lo : -1;
                            p.out.recv_topk_weights[n * K + k2] = on ? wk[k2] : 0.0f;
                        }
                    }
                }
            }
            const uint32_t *m = s_mask + e * kXWords;
            int pos = s_excl[e] + __popc(m[warp] & below);
            for (int w = 0; w < warp; ++w) pos += __popc(m[w]);
            const int64_t g = static_cast<int64_t>(eoff[b]) + pos;
            if (g < 0 || g >= p.rows_cap) {
                set_error(p.dev.err, EP_ERR_CAPACITY);
                continue;
            }
            p.out.expert_rows[g] = static_cast<int32_t>(n);
        }
    }
}

template <int KMAX, int TILE>
cudaError_t set_smem_limit(size_t bytes) {
    return cudaFuncSetAttribute(expert_layout_kernel<KMAX, TILE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

int expert_tile(int E) { return E <= kXLargeMaxE ? kXTileLarge : kXTileSmall; }
size_t expert_smem_bytes(int E) { return static_cast<size_t>(E) * (expert_tile(E) / 32 + 1) * 4; }

}  // namespace

ep_status plan_expert_layout(ep_ctx *h) {
    const int64_t T = static_cast<int64_t>(h->cfg.num_ranks) * h->cfg.tokens_per_rank;
    const int E = h->cfg.num_experts, tile = expert_tile(E);
    h->xtiles = static_cast<int>((T + tile - 1) / tile);
    const size_t smem = expert_smem_bytes(E);
    if (smem > 48 * 1024) {
        const bool k8 = h->cfg.topk <= 8;
        const cudaError_t e = tile == kXTileLarge ? (k8 ? set_smem_limit<8, kXTileLarge>(smem)
                                                        : set_smem_limit<32, kXTileLarge>(smem))
                                                  : (k8 ? set_smem_limit<8, kXTileSmall>(smem)
                                                        : set_smem_limit<32, kXTileSmall>(smem));
        if (e != cudaSuccess) return EP_ERR_CUDA;
    }
    return EP_OK;
}

ep_status launch_expert_layout(ep_ctx *h, const int32_t *topk_idx, const float *topk_weights,
                               const ep_layout_out *lay, const ep_expert_layout_out *out,
                               int64_t recv_rows, int64_t rows_cap, cudaStream_t st) {
    ExpertParams p{};
    p.topk_idx = topk_idx;
    p.topk_weights = topk_weights;
    p.token_slot = lay->token_slot;
    p.recv_base = lay->recv_base;
    p.expert_off = lay->expert_off;
    p.out = *out;
    p.dev = h->dev;
    p.R = h->cfg.num_ranks;
    p.E = h->cfg.num_experts;
    p.K = h->cfg.topk;
    p.Er = p.E / p.R;
    p.T = static_cast<int64_t>(p.R) * h->cfg.tokens_per_rank;
    p.recv_rows = recv_rows;
    p.rows_cap = rows_cap;
    p.timeout_ns = h->cfg.timeout_ns;
    p.tiles = h->xtiles;
    const uintptr_t a = reinterpret_cast<uintptr_t>(out->recv_topk_idx) |
                        reinterpret_cast<uintptr_t>(out->recv_topk_weights);
    p.vec4 = (p.K % 4 == 0 && a % 16 == 0) ? 1 : 0;
    p.vec8 = (p.K % 8 == 0 && a % 32 == 0) ? 1 : 0;
    const size_t smem = expert_smem_bytes(p.E);
    if (expert_tile(p.E) == kXTileLarge) {
        if (p.K <= 8)
            expert_layout_kernel<8, kXTileLarge><<<h->xtiles, kXTileLarge, smem, st>>>(p);
        else
            expert_layout_kernel<32, kXTileLarge><<<h->xtiles, kXTileLarge, smem, st>>>(p);
    } else {
        if (p.K <= 8)
            expert_layout_kernel<8, kXTileSmall><<<h->xtiles, kXTileSmall, smem, st>>>(p);
        else
            expert_layout_kernel<32, kXTileSmall><<<h->xtiles, kXTileSmall, smem, st>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace ep
