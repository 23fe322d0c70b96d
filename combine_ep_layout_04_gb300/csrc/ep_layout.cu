// ep_layout.cu -- token layout of one EP layer in a single pass (sm_103a).
//
// What it computes (the token-level routing bookkeeping of EP dispatch; UCCL-EP
// article s1 "fine-grained token-level communication"; a layout/rank mismatch
// is a named EP failure class in the GPU communication notes' software-stack
// table):
//   num_tokens_per_expert[s][e], is_token_in_rank[t][d], token_slot[t][d] =
//   #{t' < t : in_rank[t'][d]}, and the small scans recv_off, send_off,
//   msg_count, recv_count, recv_base, expert_off (definitions in include/ep.h).
//
// How: one CTA per tile of 256 tokens (one token per thread), tiles handed out
// in launch order by a ticket counter so every tile's predecessors are
// already running.  Per tile:
//   1. read the K picks of each token; per-token rank mask; a histogram of
//      picks per (source rank, expert) in shared memory (or, when the tile
//      spans too many ranks, warp-aggregated global atomics via match_any);
//   2. per destination column d: a warp ballot gives each token's position
//      among the warp's members of d; warp totals give the tile aggregate;
//   3. decoupled look-back (Merrill & Garland, "Single-pass Parallel Prefix
//      Scan with Decoupled Look-back", 2016), one thread per column: publish
//      the aggregate, walk back over predecessors' aggregates until an
//      inclusive prefix is found, publish the inclusive prefix.  A descriptor
//      is one 64-bit word {epoch:30 | flag:2 | value:32}; the epoch is derived
//      from the ticket, so stale words from earlier calls are never taken and
//      nothing has to be reset between calls (CUDA-graph safe);
//   4. write, at each source rank's first token, the column prefix (from
//      which the last tile derives the per-(s, d) counts and all the small
//      scans) and add the tile's histogram; fence; count the tile done;
//   5. write token_slot (lane = column, coalesced) -- after the fence, which
//      therefore does not wait for these stores; the last tile to finish
//      then runs the small scans.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kTile = 256;
constexpr int kWarps = kTile / 32;
constexpr int kHistCap = 4096;             // shared-memory histogram bins
constexpr unsigned kFull = 0xffffffffu;

// Exclusive scan of s[0, n) in place by the whole block (blockDim == kTile):
// each thread scans a run of consecutive items, warps scan the run totals with
// shuffles, one warp scans the warp totals.  Returns the total.  `tmp` holds
// at least kWarps + 1 ints.
__device__ int block_excl_scan(int *s, int n, int *tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kTile - 1) / kTile;
    const int b = tid * per, e = min(n, b + per);
    int local = 0;
    for (int i = b; i < e; ++i) local += s[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < kWarps ? tmp[lane] : 0;
        int wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kWarps) tmp[lane] = wi - v;
        if (lane == kWarps - 1) tmp[kWarps] = wi;
    }
    __syncthreads();
    int run = tmp[warp] + incl - local;
    for (int i = b; i < e; ++i) {
        const int v = s[i];
        s[i] = run;
        run += v;
    }
    const int total = tmp[kWarps];
    __syncthreads();
    return total;
}

// The last tile to finish: counts and small scans from the column prefixes
// and the histogram scratch; leaves the scratch zeroed for the next call.
__device__ void finish_layout(const LayoutParams &p, int *s_work, int *s_tmp) {
    const int tid = threadIdx.x;
    const int R = p.R, E = p.E, G = p.G;
    const int32_t *P = p.dev.col_prefix;
    // per-(s, d) counts, window offsets, message counts: every load issued
    // before the first store (P[i] and P[i + R] are the prefixes of (s, d)
    // at the first tokens of ranks s and s + 1)
    constexpr int kPairsPerThread = kMaxRanks * kMaxRanks / kTile;
    int pa[kPairsPerThread], pb[kPairsPerThread];
#pragma unroll
    for (int q = 0; q < kPairsPerThread; ++q) {
        const int i = tid + q * kTile;
        if (i < R * R) {
            pa[q] = __ldcg(P + i);
            pb[q] = __ldcg(P + i + R);
        }
    }
#pragma unroll
    for (int q = 0; q < kPairsPerThread; ++q) {
        const int i = tid + q * kTile;
        if (i >= R * R) break;
        const int c = pb[q] - pa[q];
        p.out.num_tokens_per_rank[i] = c;
        p.out.recv_off[i] = pa[q];
        p.out.msg_count[i] = (c + G - 1) / G;
        s_work[i] = c;
    }
    __syncthreads();
    block_excl_scan(s_work, R * R, s_tmp);   // row-major send order
    for (int i = tid; i < R * R; i += kTile) p.out.send_off[i] = s_work[i];
    // window sizes and starts (one warp)
    if (tid < 32) {
        int64_t run = 0;
        for (int d0 = 0; d0 < R; d0 += 32) {
            const int d = d0 + tid;
            const int c = d < R ? __ldcg(P + R * R + d) : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (tid >= o) incl += y;
            }
            if (d < R) {
                p.out.recv_count[d] = c;
                p.out.recv_base[d] = static_cast<int32_t>(run + incl - c);
            }
            run += __shfl_sync(kFull, incl, 31);
        }
        if (tid == 0) *p.dev.n_recv = run;
    }
    __syncthreads();
    // expert totals: each thread sums one expert over the source ranks,
    // copying the histogram out and clearing the scratch as it goes
    for (int e = tid; e < E; e += kTile) {
        int tot = 0;
        for (int s0 = 0; s0 < R; s0 += 8) {   // eight loads in flight, then their stores
            int v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                v[q] = s0 + q < R ? __ldcg(p.dev.hist + static_cast<int64_t>(s0 + q) * E + e) : 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (s0 + q >= R) break;
                p.out.num_tokens_per_expert[static_cast<int64_t>(s0 + q) * E + e] = v[q];
                p.dev.hist[static_cast<int64_t>(s0 + q) * E + e] = 0;
                tot += v[q];
            }
        }
        s_work[e] = tot;
    }
    __syncthreads();
    block_excl_scan(s_work, E, s_tmp);
    for (int e = tid; e < E; e += kTile) p.out.expert_off[e] = s_work[e];
    if (tid == 0) *p.dev.done = 0u;
}

__global__ void __launch_bounds__(kTile) layout_kernel(const LayoutParams p) {
    __shared__ int s_wcnt[kWarps][kMaxRanks];
    __shared__ int s_excl[kMaxRanks];
    __shared__ int s_agg[kMaxRanks];
    __shared__ int s_hist[kHistCap];
    __shared__ int s_tmp[kTile + 1];
    __shared__ unsigned long long s_ticket;
    __shared__ int s_is_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = p.R, E = p.E, K = p.K, Er = p.Er, Tpr = p.Tpr;

    if (tid == 0) s_ticket = atomicAdd(p.dev.ticket, 1ull);
    __syncthreads();
    const unsigned long long ticket = s_ticket;
    const int tile = static_cast<int>(ticket % static_cast<unsigned long long>(p.tiles));
    const uint32_t epoch = static_cast<uint32_t>((ticket / p.tiles) % ((1u << 30) - 1u)) + 1u;

    const int64_t t0 = static_cast<int64_t>(tile) * kTile;
    const int nt = static_cast<int>(min(static_cast<int64_t>(kTile), p.T - t0));
    const int s_first = static_cast<int>(t0 / Tpr);
    const int s_last = static_cast<int>((t0 + nt - 1) / Tpr);
    const int span = s_last - s_first + 1;
    const bool smem_hist = span * E <= kHistCap;
    if (smem_hist)
        for (int i = tid; i < span * E; i += kTile) s_hist[i] = 0;
    __syncthreads();

    // 1. picks -> rank mask and histogram
    const int64_t t = t0 + tid;
    const bool valid = tid < nt;
    const int s_tok = valid ? static_cast<int>(t / Tpr) : 0;
    unsigned long long mask = 0ull;
    for (int k = 0; k < K; ++k) {
        int e = valid ? __ldg(p.topk_idx + t * K + k) : -1;
        if (e < -1 || e >= E) {
            set_error(p.dev.err, EP_ERR_INVALID_ARG);
            e = -1;
        }
        if (e >= 0) mask |= 1ull << (e / Er);
        if (smem_hist) {
            if (e >= 0) atomicAdd(&s_hist[(s_tok - s_first) * E + e], 1);
        } else {
            const int key = e >= 0 ? s_tok * E + e : -1;
            const unsigned peers = __match_any_sync(kFull, key);
            if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(p.dev.hist + key, __popc(peers));
        }
    }

    // is_token_in_rank row of this token
    if (valid) {
        uint8_t *row = p.out.is_token_in_rank + t * R;
        if (p.in_rank_vec == 16) {
            for (int d = 0; d < R; d += 16) {
                uint32_t w[4];
                for (int q = 0; q < 4; ++q) {
                    uint32_t v = 0;
                    for (int b = 0; b < 4; ++b) v |= static_cast<uint32_t>((mask >> (d + 4 * q + b)) & 1ull) << (8 * b);
                    w[q] = v;
                }
                *reinterpret_cast<uint4 *>(row + d) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else if (p.in_rank_vec == 4) {
            for (int d = 0; d < R; d += 4) {
                uint32_t v = 0;
                for (int b = 0; b < 4; ++b) v |= static_cast<uint32_t>((mask >> (d + b)) & 1ull) << (8 * b);
                *reinterpret_cast<uint32_t *>(row + d) = v;
            }
        } else {
            for (int d = 0; d < R; ++d) row[d] = static_cast<uint8_t>((mask >> d) & 1ull);
        }
    }

    // 2. per-column ballots: lane j of each 32-column group keeps column j's bits
    const int ngroups = (R + 31) / 32;
    unsigned colbits[kMaxRanks / 32];
#pragma unroll
    for (int g = 0; g < kMaxRanks / 32; ++g) {
        colbits[g] = 0u;
        if (g < ngroups) {
            const int ncol = min(32, R - g * 32);
            for (int j = 0; j < ncol; ++j) {
                const unsigned b = __ballot_sync(kFull, (mask >> (g * 32 + j)) & 1ull);
                if (lane == j) colbits[g] = b;
            }
            const int d = g * 32 + lane;
            if (d < R) s_wcnt[warp][d] = __popc(colbits[g]);
        }
    }
    __syncthreads();
    if (tid < R) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int v = s_wcnt[w][tid];
            s_wcnt[w][tid] = run;
            run += v;
        }
        s_agg[tid] = run;
    }
    __syncthreads();

    // 3. decoupled look-back, one thread per column
    if (tid < R) {
        const int d = tid;
        const int agg = s_agg[d];
        unsigned long long *mine = p.dev.tile_desc + static_cast<int64_t>(tile) * R + d;
        int excl = 0;
        if (tile == 0) {
            st_relaxed(mine, look_desc(epoch, kLookPrefix, static_cast<uint32_t>(agg)));
        } else {
            st_relaxed(mine, look_desc(epoch, kLookAggregate, static_cast<uint32_t>(agg)));
            excl = lookback_excl(p.dev.tile_desc, R, d, tile, epoch, globaltimer_ns(), kDefaultTimeoutNs, p.dev.err);
            st_relaxed(mine, look_desc(epoch, kLookPrefix, static_cast<uint32_t>(excl + agg)));
        }
        s_excl[d] = excl;
        if (tile == p.tiles - 1) p.dev.col_prefix[R * R + d] = excl + agg;
    }
    __syncthreads();

    // 4. the column prefix at the first token of each source rank that
    //    starts in this tile, and the tile's histogram: the last tile reads
    //    both, so they go out before the fence
#pragma unroll
    for (int g = 0; g < kMaxRanks / 32; ++g) {
        const int d = g * 32 + lane;
        if (g >= ngroups || d >= R) continue;
        const unsigned bits = colbits[g];
        const int base = s_excl[d] + s_wcnt[warp][d];
        for (int64_t s = (t0 + Tpr - 1) / Tpr; s * Tpr < t0 + nt; ++s) {
            const int j = static_cast<int>(s * Tpr - t0) - warp * 32;
            if (j < 0 || j >= 32) continue;
            p.dev.col_prefix[s * R + d] = base + __popc(bits & ((1u << j) - 1u));
        }
    }
    if (smem_hist) {
        __syncthreads();
        for (int i = tid; i < span * E; i += kTile) {
            const int v = s_hist[i];
            if (v) atomicAdd(p.dev.hist + static_cast<int64_t>(s_first) * E + i, v);
        }
    }

    // 5. count this tile done; the last one to finish derives the small scans
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(p.dev.done, 1u) == static_cast<unsigned>(p.tiles - 1));

    // 6. token_slot, lane = column (nothing in this kernel reads it back, so
    //    the fence above does not wait for these stores)
#pragma unroll
    for (int g = 0; g < kMaxRanks / 32; ++g) {
        const int d = g * 32 + lane;
        if (g >= ngroups || d >= R) continue;
        const unsigned bits = colbits[g];
        const int base = s_excl[d] + s_wcnt[warp][d];
        for (int j = 0; j < 32; ++j) {
            const int local = warp * 32 + j;
            if (local >= nt) break;
            const int64_t tt = t0 + local;
            p.out.token_slot[tt * R + d] = ((bits >> j) & 1u) ? base + __popc(bits & ((1u << j) - 1u)) : -1;
        }
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    finish_layout(p, s_hist, s_tmp);
}

}  // namespace

ep_status launch_layout(ep_ctx *h, const int32_t *topk_idx, const ep_layout_out *out, cudaStream_t st) {
    LayoutParams p{};
    p.topk_idx = topk_idx;
    p.out = *out;
    p.dev = h->dev;
    p.R = h->cfg.num_ranks;
    p.Tpr = h->cfg.tokens_per_rank;
    p.T = static_cast<int64_t>(p.R) * p.Tpr;
    p.E = h->cfg.num_experts;
    p.K = h->cfg.topk;
    p.Er = p.E / p.R;
    p.G = h->G;
    p.tiles = h->tiles;
    const uintptr_t a = reinterpret_cast<uintptr_t>(out->is_token_in_rank);
    p.in_rank_vec = (p.R % 16 == 0 && a % 16 == 0) ? 16 : (p.R % 4 == 0 && a % 4 == 0) ? 4 : 1;
    layout_kernel<<<h->tiles, kTile, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace ep

// ---------------------------------------------------------------------------
// ep_layout_static: the layout above, for callers that cannot allocate device
// memory.  Its scratch (the look-back descriptors, the histogram, the column
// prefixes, the counters and the error word) is one file-scope device array
// of fixed size instead of a handle's cudaMalloc.  Every call on a device
// shares that array.
#include <mutex>

namespace ep {

bool ptr_usable_on(int device, const void *p);   // ep_api.cu: may the kernels dereference p?

namespace {

constexpr int kStaticMaxTokens = 262144;   // T = num_ranks * tokens_per_rank
constexpr int kStaticMaxRanks = 64;
constexpr int kStaticMaxExperts = 1024;
constexpr int kStaticMaxTiles = kStaticMaxTokens / 256;
// byte offsets inside the array (each 256-byte aligned)
constexpr size_t kSErr = 0, kSTicket = 256, kSDone = 512, kSNRecv = 768, kSPrefix = 1024;
constexpr size_t kSHist = kSPrefix + ((static_cast<size_t>(kStaticMaxRanks + 1) * kStaticMaxRanks * 4 + 255) / 256) * 256;
constexpr size_t kSDesc = kSHist + static_cast<size_t>(kStaticMaxRanks) * kStaticMaxExperts * 4;
constexpr size_t kSBytes = kSDesc + static_cast<size_t>(kStaticMaxTiles) * kStaticMaxRanks * 8;   // about 785 KB

static __device__ __align__(256) unsigned char g_layout_scratch[kSBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device, looked up once
// per device.  In host code the array's name is only a stand-in, never a
// device address.
ep_status static_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_layout_scratch) != cudaSuccess || !ptr) return EP_ERR_CUDA;
        g_static_addr[dev] = ptr;
    }
    *out = g_static_addr[dev];
    return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" ep_status ep_layout_static(const ep_config *cfg, const int32_t *topk_idx, const ep_layout_out *out,
                                      int64_t *n_recv_host, void *stream) {
    using namespace ep;
    if (!cfg || !topk_idx || !out || !out->num_tokens_per_expert || !out->num_tokens_per_rank ||
        !out->is_token_in_rank || !out->token_slot || !out->recv_off || !out->send_off || !out->msg_count ||
        !out->recv_count || !out->recv_base || !out->expert_off)
        return EP_ERR_INVALID_ARG;
    const ep_status chk = ep_config_check(cfg);
    if (chk != EP_OK) return chk;
    const int64_t T = static_cast<int64_t>(cfg->num_ranks) * cfg->tokens_per_rank;
    if (T > kStaticMaxTokens || cfg->num_ranks > kStaticMaxRanks || cfg->num_experts > kStaticMaxExperts)
        return EP_ERR_CAPACITY;   // beyond what the fixed scratch holds
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
        const void *ptrs[] = {topk_idx, out->num_tokens_per_expert, out->num_tokens_per_rank, out->is_token_in_rank,
                              out->token_slot, out->recv_off, out->send_off, out->msg_count, out->recv_count,
                              out->recv_base, out->expert_off};
        for (const void *q : ptrs)
            if (!ptr_usable_on(dev, q)) return EP_ERR_INVALID_ARG;
    }
    void *base = nullptr;
    const ep_status st0 = static_scratch(&base);
    if (st0 != EP_OK) return st0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *b = static_cast<unsigned char *>(base);
    LayoutParams p{};
    p.topk_idx = topk_idx;
    p.out = *out;
    p.R = cfg->num_ranks;
    p.Tpr = cfg->tokens_per_rank;
    p.T = T;
    p.E = cfg->num_experts;
    p.K = cfg->topk;
    p.Er = p.E / p.R;
    p.G = cfg->rows_per_msg ? cfg->rows_per_msg : default_rows_per_msg(cfg->hidden);
    p.tiles = static_cast<int>((T + 255) / 256);
    p.dev.err = reinterpret_cast<int32_t *>(b + kSErr);
    p.dev.ticket = reinterpret_cast<unsigned long long *>(b + kSTicket);
    p.dev.done = reinterpret_cast<unsigned int *>(b + kSDone);
    p.dev.n_recv = reinterpret_cast<int64_t *>(b + kSNRecv);
    p.dev.col_prefix = reinterpret_cast<int32_t *>(b + kSPrefix);
    p.dev.hist = reinterpret_cast<int32_t *>(b + kSHist);
    p.dev.tile_desc = reinterpret_cast<unsigned long long *>(b + kSDesc);
    const uintptr_t a = reinterpret_cast<uintptr_t>(out->is_token_in_rank);
    p.in_rank_vec = (p.R % 16 == 0 && a % 16 == 0) ? 16 : (p.R % 4 == 0 && a % 4 == 0) ? 4 : 1;
    // The array keeps the last call's contents: clear what this call needs at
    // zero (counters, error word, histogram, look-back descriptors).
    if (cudaMemsetAsync(b, 0, kSPrefix, st) != cudaSuccess ||
        cudaMemsetAsync(b + kSHist, 0, static_cast<size_t>(p.R) * p.E * 4, st) != cudaSuccess ||
        cudaMemsetAsync(b + kSDesc, 0, static_cast<size_t>(p.tiles) * p.R * 8, st) != cudaSuccess)
        return EP_ERR_CUDA;
    layout_kernel<<<p.tiles, kTile, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
    if (!n_recv_host) return EP_OK;
    int64_t n = 0;
    int32_t code = 0;
    if (cudaMemcpyAsync(&n, p.dev.n_recv, sizeof(n), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(&code, p.dev.err, sizeof(code), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return EP_ERR_CUDA;
    if (code != 0) return static_cast<ep_status>(code);
    *n_recv_host = n;
    return EP_OK;
}

