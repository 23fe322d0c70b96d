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
// How: one CTA per tile of 256, 512 or 1024 tokens (one token per thread; the
// tile grows with T so that large layers take about 128 tiles), tiles handed
// out in launch order by a ticket counter so every tile's predecessors are
// already running.  Per tile:
//   1. read the K picks of each token (16-byte loads when K % 4 == 0); per-token
//      rank mask; a histogram of picks per (source rank, expert) in shared
//      memory (or, when the tile spans too many ranks, warp-aggregated global
//      atomics via match_any); the token's is_token_in_rank row;
//   2. per destination column d: one warp ballot per column gives each
//      token's position among its warp's members of d; a shuffle scan over
//      the warps' counts gives each warp's offset and the tile's aggregate;
//   3. the tile publishes its aggregates (one 64-bit word per column,
//      {epoch:30 | flag:2 | value:32}; the epoch comes from the ticket, so
//      stale words of earlier calls are never taken and nothing is reset
//      between calls) and reads the aggregates of all its predecessors at
//      once, every thread taking some (predecessor, column) pairs: one round
//      trip instead of a walk.  With more than kAllPredMax tiles it falls back
//      to decoupled look-back (Merrill & Garland, "Single-pass Parallel
//      Prefix Scan with Decoupled Look-back", 2016), one thread per column;
//   4. writes, at each source rank's first token, the column prefix (from
//      which the last tile derives the per-(s, d) counts and all the small
//      scans) and adds its histogram; fence; counts the tile done;
//   5. writes token_slot, each thread its token's row in 16-byte stores --
//      after the fence, which therefore does not wait for these stores.
// One more CTA, the finisher (it draws the call's last ticket), waits until
// every tile has counted itself done, brings the column prefixes and the
// histogram into shared memory with bulk copies, and runs the small scans.
#include <atomic>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kMaxTile = 1024;
constexpr int kMaxWarps = kMaxTile / 32;
constexpr int kHistCap = 4096;             // shared-memory histogram bins
constexpr int kAllPredMax = 512;           // tiles up to which each tile sums all predecessors
constexpr int kFinHistCap = 16384;         // R x E histograms the last tile stages in shared memory
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scans of a[0, na) and b[0, nb) in place by the whole block, in
// the same passes: each thread scans a run of consecutive items of each, warps
// scan the run totals with shuffles, warps 0 and 1 scan the warp totals.
// `tmp` holds at least 2 * kMaxWarps ints.
__device__ void block_excl_scan2(int *a, int na, int *b, int nb, int *tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, bd = blockDim.x, nw = bd >> 5;
    const int pa = (na + bd - 1) / bd, pb = (nb + bd - 1) / bd;
    const int a0 = min(na, tid * pa), a1 = min(na, a0 + pa), b0 = min(nb, tid * pb), b1 = min(nb, b0 + pb);
    int la = 0, lb = 0;
    for (int i = a0; i < a1; ++i) la += a[i];
    for (int i = b0; i < b1; ++i) lb += b[i];
    int ia = la, ib = lb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(kFull, ia, o), yb = __shfl_up_sync(kFull, ib, o);
        if (lane >= o) {
            ia += ya;
            ib += yb;
        }
    }
    if (lane == 31) {
        tmp[warp] = ia;
        tmp[kMaxWarps + warp] = ib;
    }
    __syncthreads();
    if (warp < 2) {
        int *tw = tmp + warp * kMaxWarps;
        const int v = lane < nw ? tw[lane] : 0;
        int wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) tw[lane] = wi - v;
    }
    __syncthreads();
    int ra = tmp[warp] + ia - la, rb = tmp[kMaxWarps + warp] + ib - lb;
    for (int i = a0; i < a1; ++i) {
        const int v = a[i];
        a[i] = ra;
        ra += v;
    }
    for (int i = b0; i < b1; ++i) {
        const int v = b[i];
        b[i] = rb;
        rb += v;
    }
    __syncthreads();
}

__host__ __device__ __forceinline__ int pad4(int n) { return (n + 3) & ~3; }

// The finisher's staging area in dynamic shared memory (ints): the column
// prefixes, the histogram (when R x E is at most kFinHistCap), the counts,
// the expert totals.  The first two are 16-byte aligned for the bulk loads.
struct FinLayout {
    int oP, oH, oC, oT, total;
    bool stage;
    __host__ __device__ FinLayout(int R, int E) {
        stage = R * E <= kFinHistCap;
        oP = 0;
        oH = pad4((R + 1) * R);
        oC = oH + (stage ? pad4(R * E) : 0);
        oT = oC + R * R;
        total = oT + E;
    }
};

// The finisher: the CTA that drew the call's last ticket.  It waits until
// every tile has counted itself done, brings the column prefixes and the
// histogram into shared memory with two bulk copies, derives the counts and
// the small scans there, and stores everything at the end; it leaves the
// histogram scratch and the done counter zeroed for the next call.
__device__ void finish_layout(const LayoutParams &p, int *fin, int *s_tmp, uint64_t *bar) {
    const int tid = threadIdx.x, bd = blockDim.x;
    const int R = p.R, E = p.E, G = p.G, RR = R * R;
    const FinLayout f(R, E);
    int *fP = fin + f.oP, *fH = fin + f.oH, *fC = fin + f.oC, *fT = fin + f.oT;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
        const uint64_t t_start = globaltimer_ns();
        uint32_t spins = 0;
        while (ld_acquire_u32(p.dev.done) < static_cast<unsigned>(p.tiles)) {
            if ((++spins & 15u) == 0u && globaltimer_ns() - t_start > kDefaultTimeoutNs) {
                set_error(p.dev.err, EP_ERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
        // the tiles' writes (generic proxy) are acquired; the bulk copies
        // below read them through the async proxy
        fence_proxy_async_global();
        // sizes rounded up to 16 bytes: both regions are followed by padding
        // in the scratch carve
        const uint32_t bP = static_cast<uint32_t>(pad4((R + 1) * R) * 4);
        const uint32_t bH = f.stage ? static_cast<uint32_t>(pad4(R * E) * 4) : 0u;
        mbar_arrive_expect_tx(bar, bP + bH);
        bulk_g2s(fP, p.dev.col_prefix, bP, bar);
        if (f.stage) bulk_g2s(fH, p.dev.hist, bH, bar);
    }
    __syncthreads();
    if (!mbar_wait_bounded(bar, 0u, nullptr, kDefaultTimeoutNs)) set_error(p.dev.err, EP_ERR_TIMEOUT);
    for (int i = tid; i < RR; i += bd) fC[i] = fP[i + R] - fP[i];
    if (f.stage) {
        for (int e = tid; e < E; e += bd) {
            int tot = 0;
            for (int s = 0; s < R; ++s) tot += fH[s * E + e];
            fT[e] = tot;
        }
    } else {
        // large R x E: each thread sums one expert from global memory
        for (int e = tid; e < E; e += bd) {
            int tot = 0;
            for (int s0 = 0; s0 < R; s0 += 8) {
                int v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    v[q] = s0 + q < R ? __ldcg(p.dev.hist + static_cast<int64_t>(s0 + q) * E + e) : 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) tot += v[q];
            }
            fT[e] = tot;
        }
    }
    __syncthreads();
    block_excl_scan2(fC, RR, fT, E, s_tmp);   // row-major send order; expert offsets
    // window sizes and starts (one warp), then every store
    if (tid < 32) {
        int64_t run = 0;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int d = g * 32 + tid;
            const int c = d < R ? fP[RR + d] : 0;
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
        if (tid == 0) {
            *p.dev.n_recv = run;
            *p.dev.done = 0u;
        }
    }
    for (int i = tid; i < RR; i += bd) {
        const int c = fP[i + R] - fP[i];
        p.out.num_tokens_per_rank[i] = c;
        p.out.recv_off[i] = fP[i];
        p.out.msg_count[i] = (c + G - 1) / G;
        p.out.send_off[i] = fC[i];
    }
    for (int e = tid; e < E; e += bd) p.out.expert_off[e] = fT[e];
    for (int i = tid; i < R * E; i += bd) {
        p.out.num_tokens_per_expert[i] = f.stage ? fH[i] : __ldcg(p.dev.hist + i);
        p.dev.hist[i] = 0;
    }
}

__global__ void __launch_bounds__(kMaxTile) layout_kernel(const LayoutParams p) {
    __shared__ __align__(16) unsigned s_ballot[kMaxWarps][kMaxRanks];   // per warp and column: members among its 32 tokens
    __shared__ __align__(16) int s_woff[kMaxWarps][kMaxRanks];          // per warp and column: members in earlier warps
    __shared__ __align__(16) int s_excl[kMaxRanks];                     // per column: members in earlier tiles
    __shared__ int s_agg[kMaxRanks];                                    // per column: members in this tile
    __shared__ int s_hist[kHistCap];
    __shared__ int s_tmp[2 * kMaxWarps];
    __shared__ unsigned long long s_mask[kMaxTile];                     // rank mask of each token of the tile
    __shared__ unsigned long long s_ticket;
    __shared__ __align__(8) uint64_t s_bar;
    extern __shared__ __align__(16) int fin[];                          // the finisher's staging

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bd = blockDim.x, nw = bd >> 5;
    const int R = p.R, E = p.E, K = p.K, Tpr = p.Tpr;

    if (tid == 0) s_ticket = atomicAdd(p.dev.ticket, 1ull);
    if (tid < R) s_excl[tid] = 0;
    __syncthreads();
    // tickets of one call: tiles 0 .. tiles-1 in order, then the finisher
    const unsigned long long ticket = s_ticket, per_call = static_cast<unsigned long long>(p.tiles) + 1ull;
    const int tile = static_cast<int>(ticket % per_call);
    const uint32_t epoch = static_cast<uint32_t>((ticket / per_call) % ((1u << 30) - 1u)) + 1u;
    if (tile == p.tiles) {
        finish_layout(p, fin, s_tmp, &s_bar);
        return;
    }

    // T < 2^31 (ep_config_check), so token numbers fit in 32 bits
    const int t0 = tile * bd;
    const int nt = min(bd, static_cast<int>(p.T) - t0);
    const int t = t0 + tid;
    const bool valid = tid < nt;
    const int s_first = t0 / Tpr;
    const int s_last = (t0 + nt - 1) / Tpr;
    const int span = s_last - s_first + 1;
    const bool smem_hist = span * E <= kHistCap;
    const int s_tok = valid ? t / Tpr : s_first;

    // 1. picks -> rank mask (the histogram waits until the aggregates are out)
    const int32_t *prow = p.topk_idx + static_cast<int64_t>(t) * K;
    unsigned long long mask = 0ull;
    for (int k0 = 0; k0 < K; k0 += 8) {
        int ev[8];
        if (p.topk_vec4 && k0 + 8 <= K) {
            const int4 a = valid ? __ldg(reinterpret_cast<const int4 *>(prow + k0)) : make_int4(-1, -1, -1, -1);
            const int4 b = valid ? __ldg(reinterpret_cast<const int4 *>(prow + k0 + 4)) : make_int4(-1, -1, -1, -1);
            ev[0] = a.x; ev[1] = a.y; ev[2] = a.z; ev[3] = a.w;
            ev[4] = b.x; ev[5] = b.y; ev[6] = b.z; ev[7] = b.w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) ev[q] = (valid && k0 + q < K) ? __ldg(prow + k0 + q) : -1;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = ev[q];
            if (e < -1 || e >= E) set_error(p.dev.err, EP_ERR_INVALID_ARG);
            else if (e >= 0) mask |= 1ull << (p.er_shift >= 0 ? (e >> p.er_shift) : (e / p.Er));
        }
    }
    s_mask[tid] = mask;
    if (smem_hist)
        for (int i = tid; i < span * E; i += bd) s_hist[i] = 0;

    // 2. per 32-column group, transpose the warp's 32 x 32 bit matrix (row =
    //    token, column = rank) in five shuffle rounds, so that lane j holds
    //    column j's bits over the warp's tokens
    const int ngroups = (R + 31) >> 5;
#pragma unroll
    for (int g = 0; g < kMaxRanks / 32; ++g) {
        if (g >= ngroups) break;
        unsigned x = static_cast<unsigned>(mask >> (32 * g));
#pragma unroll
        for (int sft = 16; sft > 0; sft >>= 1) {
            const unsigned m = sft == 16 ? 0x0000FFFFu : sft == 8 ? 0x00FF00FFu : sft == 4 ? 0x0F0F0F0Fu
                             : sft == 2 ? 0x33333333u : 0x55555555u;
            const unsigned y = __shfl_xor_sync(kFull, x, sft);
            x = (lane & sft) ? ((x & ~m) | ((y & ~m) >> sft)) : ((x & m) | ((y & m) << sft));
        }
        if (g * 32 + lane < R) s_ballot[warp][g * 32 + lane] = x;
    }
    __syncthreads();
    // per column: warps' member counts scanned across the warps
    for (int d = warp; d < R; d += nw) {
        const int c = lane < nw ? __popc(s_ballot[lane][d]) : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < nw) s_woff[lane][d] = incl - c;
        if (lane == 31) s_agg[d] = incl;
    }
    __syncthreads();

    // 3. publish this tile's aggregates; the histogram of the picks (read again,
    //    from cache); then the predecessors' aggregates
    unsigned long long *desc = p.dev.tile_desc;
    const bool all_pred = p.tiles <= kAllPredMax;
    if (tid < R)
        st_relaxed(desc + static_cast<int64_t>(tile) * R + tid,
                   look_desc(epoch, (tile == 0 && !all_pred) ? kLookPrefix : kLookAggregate,
                             static_cast<uint32_t>(s_agg[tid])));
    for (int k = 0; k < K; ++k) {
        int e = valid ? __ldg(prow + k) : -1;
        if (e < -1 || e >= E) e = -1;
        if (smem_hist) {
            if (e >= 0) atomicAdd(&s_hist[(s_tok - s_first) * E + e], 1);
        } else {
            const int key = e >= 0 ? s_tok * E + e : -1;
            const unsigned peers = __match_any_sync(kFull, key);
            if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(p.dev.hist + key, __popc(peers));
        }
    }
    if (tile > 0) {
        const uint64_t t_start = globaltimer_ns();
        if (all_pred) {
            // thread tid takes column tid % R of predecessors tid / R, + step, ...
            const int step = bd / R;
            const int d = tid % R, j0 = tid / R;
            if (j0 < step) {
                int sum = 0;
                for (int jb = j0; jb < tile; jb += 8 * step) {
                    unsigned long long v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int j = jb + q * step;
                        v[q] = j < tile ? ld_relaxed(desc + static_cast<int64_t>(j) * R + d) : 0ull;
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int j = jb + q * step;
                        if (j >= tile) break;
                        unsigned long long x = v[q];
                        uint32_t spins = 0;
                        while (static_cast<uint32_t>(x >> 34) != epoch || ((x >> 32) & 3u) != kLookAggregate) {
                            if ((++spins & 15u) == 0u && globaltimer_ns() - t_start > kDefaultTimeoutNs) {
                                set_error(p.dev.err, EP_ERR_TIMEOUT);
                                x = 0ull;
                                break;
                            }
                            __nanosleep(32);
                            x = ld_relaxed(desc + static_cast<int64_t>(j) * R + d);
                        }
                        sum += static_cast<int>(static_cast<uint32_t>(x));
                    }
                }
                if (sum) atomicAdd(&s_excl[d], sum);
            }
        } else if (tid < R) {
            const int excl = lookback_excl(desc, R, tid, tile, epoch, t_start, kDefaultTimeoutNs, p.dev.err);
            s_excl[tid] = excl;
            st_relaxed(desc + static_cast<int64_t>(tile) * R + tid,
                       look_desc(epoch, kLookPrefix, static_cast<uint32_t>(excl + s_agg[tid])));
        }
    }
    __syncthreads();

    // 4. what the finisher reads -- the column prefix at the first token of
    //    each source rank that starts here, the column totals (last tile by
    //    position) and the histogram -- goes out before the fence
    const unsigned lt = lanemask_lt();
    if (tile == p.tiles - 1 && tid < R) p.dev.col_prefix[R * R + tid] = s_excl[tid] + s_agg[tid];
    if (valid && t == s_tok * Tpr) {
        int32_t *pr = p.dev.col_prefix + static_cast<int64_t>(s_tok) * R;
        for (int d = 0; d < R; ++d) pr[d] = s_excl[d] + s_woff[warp][d] + __popc(s_ballot[warp][d] & lt);
    }
    if (smem_hist) {
        for (int i = tid; i < span * E; i += bd) {
            const int v = s_hist[i];
            if (v) atomicAdd(p.dev.hist + static_cast<int64_t>(s_first) * E + i, v);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) atomicAdd(p.dev.done, 1u);

    // 5. the tile's rows of is_token_in_rank and token_slot, last: no barrier
    //    follows them.  A warp's 32 rows are contiguous; each lane stores
    //    16-byte pieces of them, so every store instruction covers whole lines.
    const int wt0 = t0 + warp * 32;                       // the warp's first token
    const int wn = max(0, min(32, nt - warp * 32));       // its tokens
    if (p.in_rank_vec == 16) {
        uint8_t *base = p.out.is_token_in_rank + static_cast<int64_t>(wt0) * R;
        for (int c = lane; c < wn * R / 16; c += 32) {    // piece c: token c*16/R, columns (c*16) % R ..
            const int j = c * 16 / R, d0 = (c * 16) % R;
            const unsigned long long m = s_mask[warp * 32 + j];
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // four mask bits -> four bytes of 0/1
                const uint32_t nib = static_cast<uint32_t>(m >> (d0 + 4 * q)) & 0xFu;
                w[q] = (nib * 0x00204081u) & 0x01010101u;
            }
            *reinterpret_cast<uint4 *>(base + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else if (valid) {
        uint8_t *row = p.out.is_token_in_rank + static_cast<int64_t>(t) * R;
        for (int d = 0; d < R; ++d) row[d] = static_cast<uint8_t>((mask >> d) & 1ull);
    }
    if (p.slot_vec) {
        int32_t *base = p.out.token_slot + static_cast<int64_t>(wt0) * R;
        for (int c = lane; c < wn * R / 4; c += 32) {     // piece c: token c*4/R, columns (c*4) % R ..
            const int j = c * 4 / R, d0 = (c * 4) % R;
            const unsigned below = (1u << j) - 1u;
            const uint4 b = *reinterpret_cast<const uint4 *>(&s_ballot[warp][d0]);
            const int4 wo = *reinterpret_cast<const int4 *>(&s_woff[warp][d0]);
            const int4 ex = *reinterpret_cast<const int4 *>(&s_excl[d0]);
            int4 v;
            v.x = ((b.x >> j) & 1u) ? ex.x + wo.x + __popc(b.x & below) : -1;
            v.y = ((b.y >> j) & 1u) ? ex.y + wo.y + __popc(b.y & below) : -1;
            v.z = ((b.z >> j) & 1u) ? ex.z + wo.z + __popc(b.z & below) : -1;
            v.w = ((b.w >> j) & 1u) ? ex.w + wo.w + __popc(b.w & below) : -1;
            *reinterpret_cast<int4 *>(base + c * 4) = v;
        }
    } else if (valid) {
        int32_t *srow = p.out.token_slot + static_cast<int64_t>(t) * R;
        for (int d = 0; d < R; ++d)
            srow[d] = ((mask >> d) & 1ull) ? s_excl[d] + s_woff[warp][d] + __popc(s_ballot[warp][d] & lt) : -1;
    }
}

}  // namespace

int layout_tile(int64_t T) { return T <= 16384 ? 256 : T <= 65536 ? 512 : kMaxTile; }

// Dynamic shared memory of the layout kernel: the finisher's staging area.
size_t layout_smem_bytes(int R, int E) { return static_cast<size_t>(FinLayout(R, E).total) * 4; }

// Allows the kernel the largest staging area any shape asks for, once per
// device (R = 64 with R x E at the staging cap is the largest).
ep_status layout_prepare() {
    constexpr int kDevs = 64;
    static std::atomic<int> ready[kDevs];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return EP_ERR_CUDA;
    if (ready[dev].load(std::memory_order_acquire)) return EP_OK;
    size_t most = 0;
    for (int R = 1; R <= kMaxRanks; ++R)
        for (int E = R; E <= 4096; E += R) most = most > layout_smem_bytes(R, E) ? most : layout_smem_bytes(R, E);
    if (cudaFuncSetAttribute(layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(most)) !=
        cudaSuccess)
        return EP_ERR_CUDA;
    ready[dev].store(1, std::memory_order_release);
    return EP_OK;
}

void fill_layout_vec(LayoutParams &p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.out.is_token_in_rank);
    p.in_rank_vec = (p.R % 16 == 0 && a % 16 == 0) ? 16 : (p.R % 4 == 0 && a % 4 == 0) ? 4 : 1;
    p.slot_vec = (p.R % 4 == 0 && reinterpret_cast<uintptr_t>(p.out.token_slot) % 16 == 0) ? 1 : 0;
    p.topk_vec4 = (p.K % 4 == 0 && reinterpret_cast<uintptr_t>(p.topk_idx) % 16 == 0) ? 1 : 0;
    p.er_shift = (p.Er & (p.Er - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(p.Er)) : -1;
}

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
    fill_layout_vec(p);
    if (layout_prepare() != EP_OK) return EP_ERR_CUDA;
    // the token tiles, plus the finisher
    layout_kernel<<<h->tiles + 1, layout_tile(p.T), layout_smem_bytes(p.R, p.E), st>>>(p);
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
    const int tile_tokens = layout_tile(T);
    p.tiles = static_cast<int>((T + tile_tokens - 1) / tile_tokens);
    p.dev.err = reinterpret_cast<int32_t *>(b + kSErr);
    p.dev.ticket = reinterpret_cast<unsigned long long *>(b + kSTicket);
    p.dev.done = reinterpret_cast<unsigned int *>(b + kSDone);
    p.dev.n_recv = reinterpret_cast<int64_t *>(b + kSNRecv);
    p.dev.col_prefix = reinterpret_cast<int32_t *>(b + kSPrefix);
    p.dev.hist = reinterpret_cast<int32_t *>(b + kSHist);
    p.dev.tile_desc = reinterpret_cast<unsigned long long *>(b + kSDesc);
    fill_layout_vec(p);
    // The array keeps the last call's contents: clear what this call needs at
    // zero (counters, error word, histogram, look-back descriptors).
    if (cudaMemsetAsync(b, 0, kSPrefix, st) != cudaSuccess ||
        cudaMemsetAsync(b + kSHist, 0, static_cast<size_t>(p.R) * p.E * 4, st) != cudaSuccess ||
        cudaMemsetAsync(b + kSDesc, 0, static_cast<size_t>(p.tiles) * p.R * 8, st) != cudaSuccess)
        return EP_ERR_CUDA;
    if (layout_prepare() != EP_OK) return EP_ERR_CUDA;
    layout_kernel<<<p.tiles + 1, tile_tokens, layout_smem_bytes(p.R, p.E), st>>>(p);
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

