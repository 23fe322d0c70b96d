// ep_dispatch.cu -- EP dispatch with TransferCmd rings (sm_103a).
//
// What it does (UCCL-EP article: s6 "Dispatch"; s2.2 the lock-free ring of
// TransferCmd records with head/tail atomics, batch enqueue of up to 8
// commands and flow control against kMaxInflight; s2.3 the TransferCmd fields
// {dst_rank, src_offset, dst_offset, size}; s3.1 Write completes when the
// target memory is visible, Drain waits until the queue is empty; s4.1 the
// pipelined DispatchKernel and packing of small tokens; s4.2 independent
// channels; NCCL GIN article s2.2.1 byte-offset windows):
//
//   for every token t and destination rank d with token_slot[t][d] >= 0:
//       recv[recv_base[d] + token_slot[t][d]] <- x[t]        (one copy per rank)
//   for every message g of pair (s, d) -- up to G consecutive rows of the pair --
//       post TransferCmd{d, rows*B, (send_off[s][d] + gG)*B, (recv_off[s][d] + gG)*B}
//       into ring d % C once all its rows have landed.
//
// How: one persistent cooperative kernel, one CTA per SM, three warps:
//   warp 0  copy warp: 1-D TMA bulk loads of token rows (a run of whole rows
//           when they are small, a piece of one row when it is large) into a
//           ring of shared-memory stages, then one TMA bulk store per
//           (row, destination) from the stage; each source row is read from
//           HBM once whatever its number of destinations.  Lane 0 issues the
//           loads; all 32 lanes issue stores, each tracking its own bulk
//           groups, so that a stage is recycled only when every lane's stores
//           from it have completed.
//   warp 1  meta/post warp: per chunk of 32 tokens of one source rank, reads
//           the token_slot rows, builds each token's destination-row list and
//           each rank's slot range for the copy warp, and -- once the copy
//           warp reports the chunk's stores complete -- works out which
//           messages the chunk completed (a message whose rows were written by
//           several CTAs is completed by whichever CTA lands its last row,
//           counted with one atomic per CTA and message) and posts them,
//           grouped per ring into batches of up to `batch` commands: reserve
//           with one atomicAdd on head, wait (bounded) while the ring would
//           exceed max_inflight, write the records, publish each slot with a
//           release store of its sequence tag.
//   warp 2  (CTAs 0..C-1) ring consumer for channel blockIdx.x: each step
//           polls every slot that can be outstanding (max_inflight of them,
//           drain_batch = 32 per warp-wide poll, all loads in flight at once),
//           retires the longest published run into the channel's log, marks
//           those slots COMPLETED and advances tail with one release store; it
//           stops when the channel's message count (from msg_count) has been
//           retired, which is the drain.
// Every wait is bounded by the handle's timeout and by the grid's error word;
// none traps.  A cooperative launch keeps all CTAs -- and so all consumers --
// resident while producers wait on them.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kThreads = 96;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kCopyWarp = 0, kMetaWarp = 1, kConsumerWarp = 2;

// Shared-memory carve, identical on host and device.
struct SmemLayout {
    int stage_off, meta_off, meta_slot_bytes, scratch_off, bar_off, total;
    // meta slot (ints): dst[32*R] | pref[33] | lo[R] | hi[R] | info[4]
    __host__ __device__ static int meta_ints(int R) { return ((32 * R + 33 + 2 * R + 4) + 3) & ~3; }
    __host__ __device__ SmemLayout(int R, int C, int stage_bytes, int stages, int meta_slots) {
        stage_off = 0;
        meta_off = stage_bytes * stages;
        meta_slot_bytes = meta_ints(R) * 4;
        scratch_off = meta_off + meta_slot_bytes * meta_slots;
        // scratch ints: rbase[R] | nd[R] | gs[R] | ctot[C] | cbb[C+1] | flags[4]
        const int scratch_ints = (3 * R + 2 * C + 1 + 4 + 3) & ~3;
        bar_off = (scratch_off + scratch_ints * 4 + 15) & ~15;
        total = bar_off + 8 * (stages + 2 * meta_slots);
    }
};

struct MetaSlot {
    int *dst, *pref, *lo, *hi, *info;   // info: chunk, ntok, src rank, first token
    __device__ MetaSlot(uint8_t *base, int R) {
        dst = reinterpret_cast<int *>(base);
        pref = dst + 32 * R;
        lo = pref + 33;
        hi = lo + R;
        info = hi + R;
    }
};

__device__ __forceinline__ int chunk_ntok(const DispatchParams &p, int k) {
    const int ci = k % p.chunks_per_rank;
    return min(kChunkTokens, p.Tpr - ci * kChunkTokens);
}
__device__ __forceinline__ int64_t chunk_tok0(const DispatchParams &p, int k) {
    const int s = k / p.chunks_per_rank, ci = k % p.chunks_per_rank;
    return static_cast<int64_t>(s) * p.Tpr + static_cast<int64_t>(ci) * kChunkTokens;
}
__device__ __forceinline__ int chunk_items(const DispatchParams &p, int ntok) {
    return p.pieces > 1 ? ntok * p.pieces : (ntok + p.rows_per_item - 1) / p.rows_per_item;
}

// Walks this CTA's items: chunks blockIdx.x, +gridDim.x, ...; items within.
struct ItemCursor {
    int m, k, q, ntok, nitems;
    bool valid;
    __device__ void start(const DispatchParams &p) {
        m = 0;
        k = blockIdx.x;
        q = 0;
        valid = k < p.nchunks;
        if (valid) {
            ntok = chunk_ntok(p, k);
            nitems = chunk_items(p, ntok);
        }
    }
    __device__ void advance(const DispatchParams &p) {
        if (++q < nitems) return;
        q = 0;
        ++m;
        k += gridDim.x;
        valid = k < p.nchunks;
        if (valid) {
            ntok = chunk_ntok(p, k);
            nitems = chunk_items(p, ntok);
        }
    }
    // tokens [ta, tb) of the chunk, byte range [off, off + len) of each row
    __device__ void geometry(const DispatchParams &p, int &ta, int &tb, int &off, int &len) const {
        if (p.pieces > 1) {
            ta = q / p.pieces;
            tb = ta + 1;
            off = (q % p.pieces) * p.piece_bytes;
            len = static_cast<int>(min(static_cast<int64_t>(p.piece_bytes), p.row_bytes - off));
        } else {
            ta = q * p.rows_per_item;
            tb = min(ntok, ta + p.rows_per_item);
            off = 0;
            len = static_cast<int>(p.row_bytes);
        }
    }
};

// ------------------------------------------------------------------ copy warp
__device__ void copy_warp(const DispatchParams &p, uint8_t *smem, const SmemLayout &L, uint64_t *bar_full,
                          uint64_t *meta_full, uint64_t *chunk_done) {
    const int lane = threadIdx.x & 31;
    const int S = p.stages, P = p.prefetch, NS = p.meta_slots;
    const int64_t B = p.row_bytes;
    ItemCursor ld, stc;
    ld.start(p);
    stc.start(p);
    int64_t n_loaded = 0, n_stored = 0;
    int stored_chunks = 0, signalled = 0;
    int64_t last_item[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // last item of in-flight chunks (NS <= 8)
    bool ok = true;

    auto issue_load = [&](const ItemCursor &c, int64_t idx) {
        if (lane == 0) {
            int ta, tb, off, len;
            c.geometry(p, ta, tb, off, len);
            const int stage = static_cast<int>(idx % S);
            const uint32_t bytes = static_cast<uint32_t>((tb - ta) * len);
            const uint8_t *src = p.x + (chunk_tok0(p, c.k) + ta) * B + off;
            mbar_arrive_expect_tx(&bar_full[stage], bytes);
            bulk_g2s(smem + L.stage_off + static_cast<int64_t>(stage) * p.stage_bytes, src, bytes, &bar_full[stage]);
        }
    };
    // Signal every stored chunk whose last item is <= upto as complete.
    auto signal_upto = [&](int64_t upto) {
        fence_proxy_async_global();
        __syncwarp();
        while (signalled < stored_chunks && last_item[signalled % NS] <= upto) {
            if (lane == 0) mbar_arrive(&chunk_done[signalled % NS]);
            ++signalled;
        }
    };

    for (int i = 0; i < P && ld.valid; ++i) {
        issue_load(ld, n_loaded++);
        ld.advance(p);
    }
    while (stc.valid) {
        const int64_t i = n_stored;
        const int slot = stc.m % NS;
        if (stc.q == 0) {
            const uint32_t par = static_cast<uint32_t>(stc.m / NS) & 1u;
            // warp-uniform decisions: a phase may complete between two lanes' tests
            if (!__all_sync(kFull, mbar_test(&meta_full[slot], par))) {
                // the meta warp may be waiting for earlier chunks: complete them first
                bulk_wait<0>();
                signal_upto(INT64_MAX);
                if (!__all_sync(kFull, mbar_wait_bounded(&meta_full[slot], par, p.dev.err, p.timeout_ns))) {
                    set_error(p.dev.err, EP_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
        const int stage = static_cast<int>(i % S);
        if (!__all_sync(kFull, mbar_wait_bounded(&bar_full[stage], static_cast<uint32_t>(i / S) & 1u, p.dev.err,
                                                 p.timeout_ns))) {
            set_error(p.dev.err, EP_ERR_TIMEOUT);
            ok = false;
            break;
        }
        {
            MetaSlot ms(smem + L.meta_off + static_cast<int64_t>(slot) * L.meta_slot_bytes, p.R);
            int ta, tb, off, len;
            stc.geometry(p, ta, tb, off, len);
            const uint8_t *stage_base = smem + L.stage_off + static_cast<int64_t>(stage) * p.stage_bytes;
            const int pb = ms.pref[ta], pe = ms.pref[tb];
            int tl = ta;
            for (int pi = pb + lane; pi < pe; pi += 32) {
                while (ms.pref[tl + 1] <= pi) ++tl;
                const int row = ms.dst[tl * p.R + (pi - ms.pref[tl])];
                bulk_s2g(p.recv + static_cast<int64_t>(row) * B + off, stage_base + static_cast<int64_t>(tl - ta) * len,
                         static_cast<uint32_t>(len));
            }
            bulk_commit();
        }
        if (stc.q == stc.nitems - 1) {
            last_item[stc.m % NS] = i;
            ++stored_chunks;
        }
        ++n_stored;
        stc.advance(p);
        if (ld.valid) {
            // stage of item n_loaded was last used by item n_loaded - S
            bulk_wait_n(S - P);
            signal_upto(n_stored - 1 - (S - P));
            issue_load(ld, n_loaded++);
            ld.advance(p);
        }
    }
    bulk_wait<0>();
    if (ok) {
        signal_upto(INT64_MAX);
    } else {
        // abort: let every load already issued land before the CTA exits (the
        // wait ignores the error word; it is still bounded by the time limit)
        for (int64_t j = n_stored; j < n_loaded; ++j)
            mbar_wait_bounded(&bar_full[j % S], static_cast<uint32_t>(j / S) & 1u, nullptr, p.timeout_ns);
        __syncwarp();
    }
}

// ------------------------------------------------------------ meta/post warp
__device__ void build_meta(const DispatchParams &p, int k, const MetaSlot &ms, const int *rbase) {
    const int lane = threadIdx.x & 31;
    const int R = p.R;
    const int ntok = chunk_ntok(p, k);
    const int64_t tok0 = chunk_tok0(p, k);
    const bool valid = lane < ntok;
    const int64_t t = tok0 + lane;
    int n = 0;
    int *dst = ms.dst + lane * R;
    for (int d0 = 0; d0 < R; d0 += 4) {
        int v[4] = {-1, -1, -1, -1};
        if (valid) {
            if (p.slot_vec) {
                const int4 q = __ldg(reinterpret_cast<const int4 *>(p.token_slot + t * R + d0));
                v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
            } else {
                for (int j = 0; j < 4 && d0 + j < R; ++j) v[j] = __ldg(p.token_slot + t * R + d0 + j);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = d0 + j;
            if (d >= R) break;
            const int sl = v[j];
            if (sl >= 0) {
                const int64_t row = static_cast<int64_t>(rbase[d]) + sl;
                if (row >= 0 && row < p.cap_rows) {
                    dst[n++] = static_cast<int>(row);
                } else {
                    set_error(p.dev.err, EP_ERR_CAPACITY);
                }
            }
            const int lo = __reduce_min_sync(kFull, sl >= 0 ? sl : INT32_MAX);
            const int hi = __reduce_max_sync(kFull, sl >= 0 ? sl : -1);
            if (lane == 0) {
                ms.lo[d] = lo == INT32_MAX ? -1 : lo;
                ms.hi[d] = hi;
            }
        }
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    ms.pref[lane] = incl - n;
    if (lane == 31) ms.pref[32] = incl;
    if (lane == 0) {
        ms.info[0] = k;
        ms.info[1] = ntok;
        ms.info[2] = k / p.chunks_per_rank;
        ms.info[3] = 0;
    }
}

// Rows of message g of a pair with cnt rows.
__device__ __forceinline__ int msg_rows(int g, int G, int cnt) { return min(G, cnt - g * G); }

// Adds `rows` landed rows to message (s, d, g); true if this call completed it.
__device__ __forceinline__ bool message_fill(const DispatchParams &p, int s, int d, int g, int rows, int need) {
    if (g < 0 || g >= p.msgs_per_pair) {
        set_error(p.dev.err, EP_ERR_INVALID_ARG);
        return false;
    }
    unsigned int *ctr = p.dev.msg_fill + (static_cast<int64_t>(s) * p.R + d) * p.msgs_per_pair + g;
    const unsigned old = atomicAdd(ctr, static_cast<unsigned>(rows));
    if (old + static_cast<unsigned>(rows) == static_cast<unsigned>(need)) {
        *ctr = 0u;   // last arrival: leave it zeroed for the next call
        __threadfence();
        return true;
    }
    return false;
}

// Posts n commands of channel c, flat indices [f0, f0 + n) of this chunk's list.
__device__ bool post_batch(const DispatchParams &p, int c, int s, int f0, int n, const int *nd, const int *gs) {
    unsigned long long *head = p.dev.head + static_cast<int64_t>(c) * kHeadStride;
    unsigned long long *tail = p.dev.tail + static_cast<int64_t>(c) * kHeadStride;
    const unsigned long long base = atomicAdd(head, static_cast<unsigned long long>(n));
    unsigned long long tl = ld_acquire(tail);
    unsigned long long stalls = 0;
    if (base + n - tl > static_cast<unsigned long long>(p.max_inflight)) {
        const uint64_t t0 = globaltimer_ns();
        unsigned sleep = 32;
        while (true) {
            __nanosleep(sleep);
            sleep = min(sleep * 2u, 1024u);
            tl = ld_acquire(tail);
            ++stalls;
            if (base + n - tl <= static_cast<unsigned long long>(p.max_inflight)) break;
            if (read_error(p.dev.err) != 0) return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                set_error(p.dev.err, EP_ERR_TIMEOUT);
                return false;
            }
        }
    }
    const int R = p.R, G = p.G, C = p.C;
    const int64_t B = p.row_bytes;
    for (int i = 0; i < n; ++i) {
        int f = f0 + i, d = c;
        while (d < R && f >= nd[d]) {
            f -= nd[d];
            d += C;
        }
        if (d >= R) {   // cannot happen with a consistent list
            set_error(p.dev.err, EP_ERR_INVALID_ARG);
            return false;
        }
        const int g = gs[d] + f;
        const int j0 = g * G;
        const int cnt = __ldg(p.cnt + s * R + d);
        const int rows = msg_rows(g, G, cnt);
        const unsigned long long idx = base + i;
        const int64_t sidx = static_cast<int64_t>(c) * p.D + static_cast<int64_t>(idx & static_cast<unsigned long long>(p.D - 1));
        uint4 *rec = reinterpret_cast<uint4 *>(p.dev.slots + sidx);
        const uint64_t src_off = static_cast<uint64_t>((static_cast<int64_t>(__ldg(p.send_off + s * R + d)) + j0) * B);
        const uint64_t dst_off = static_cast<uint64_t>((static_cast<int64_t>(__ldg(p.recv_off + s * R + d)) + j0) * B);
        rec[0] = make_uint4(static_cast<uint32_t>(d), static_cast<uint32_t>(rows * B), static_cast<uint32_t>(src_off),
                            static_cast<uint32_t>(src_off >> 32));
        rec[1] = make_uint4(static_cast<uint32_t>(dst_off), static_cast<uint32_t>(dst_off >> 32), 0u, 0u);
        st_release(p.dev.status + sidx, 2ull * idx + 1ull);
    }
    RingStatsDev *stt = p.dev.stats + c;
    atomicAdd(&stt->batches, 1ull);
    atomicMax(&stt->max_batch, static_cast<unsigned>(n));
    atomicMax(&stt->max_inflight, static_cast<unsigned>(base + n - tl));
    if (stalls) atomicAdd(&stt->stall_polls, stalls);
    return true;
}

// After the chunk's rows have landed: the chunk's completed messages, posted.
__device__ bool post_chunk(const DispatchParams &p, const MetaSlot &ms, int *nd, int *gs, int *ctot, int *cbb) {
    const int lane = threadIdx.x & 31;
    const int R = p.R, C = p.C, G = p.G;
    const int s = ms.info[2];
    __threadfence();   // this CTA's rows are visible before any count or record
    for (int d = lane; d < R; d += 32) {
        const int lo = ms.lo[d], hi = ms.hi[d];
        int n = 0, g_start = 0;
        if (hi >= 0) {
            const int ro = __ldg(p.recv_off + s * R + d);
            const int cnt = __ldg(p.cnt + s * R + d);
            const int jlo = lo - ro, jhi = hi - ro;
            if (jlo < 0 || jhi < jlo || jhi >= cnt) {
                set_error(p.dev.err, EP_ERR_INVALID_ARG);
            } else {
                const int ga = jlo / G, gb = jhi / G;
                int m0 = ga * G, m1 = m0 + msg_rows(ga, G, cnt) - 1;
                int in_lo = max(m0, jlo), in_hi = min(m1, jhi);
                bool done = (in_lo == m0 && in_hi == m1) ||
                            message_fill(p, s, d, ga, in_hi - in_lo + 1, m1 - m0 + 1);
                g_start = done ? ga : ga + 1;
                int g_end = ga + 1;
                if (gb > ga) {
                    m0 = gb * G;
                    m1 = m0 + msg_rows(gb, G, cnt) - 1;
                    in_hi = min(m1, jhi);
                    done = (in_hi == m1) || message_fill(p, s, d, gb, in_hi - m0 + 1, m1 - m0 + 1);
                    g_end = done ? gb + 1 : gb;
                }
                n = max(0, g_end - g_start);
            }
        }
        nd[d] = n;
        gs[d] = g_start;
    }
    __syncwarp();
    for (int c = lane; c < C; c += 32) {
        int tot = 0;
        for (int d = c; d < R; d += C) tot += nd[d];
        ctot[c] = tot;
    }
    __syncwarp();
    if (lane == 0) {
        int run = 0;
        for (int c = 0; c < C; ++c) {
            cbb[c] = run;
            run += (ctot[c] + p.batch - 1) / p.batch;
        }
        cbb[C] = run;
    }
    __syncwarp();
    const int nb = cbb[C];
    bool ok = true;
    for (int b = lane; b < nb; b += 32) {
        int c = 0;
        while (cbb[c + 1] <= b) ++c;
        const int f0 = (b - cbb[c]) * p.batch;
        const int n = min(p.batch, ctot[c] - f0);
        if (!post_batch(p, c, s, f0, n, nd, gs)) {
            ok = false;
            break;
        }
    }
    return __all_sync(kFull, ok);
}

__device__ void meta_warp(const DispatchParams &p, uint8_t *smem, const SmemLayout &L, uint64_t *meta_full,
                          uint64_t *chunk_done, int *scratch) {
    const int lane = threadIdx.x & 31;
    const int R = p.R, C = p.C, NS = p.meta_slots;
    int *rbase = scratch, *nd = scratch + R, *gs = scratch + 2 * R, *ctot = scratch + 3 * R, *cbb = ctot + C;
    auto slot_of = [&](int m) {
        return MetaSlot(smem + L.meta_off + static_cast<int64_t>(m % NS) * L.meta_slot_bytes, R);
    };
    int n_my = 0;
    for (int m = 0;; ++m) {
        const int k = blockIdx.x + m * gridDim.x;
        if (k >= p.nchunks) break;
        n_my = m + 1;
        if (m >= NS) {
            const int mm = m - NS;
            if (!__all_sync(kFull, mbar_wait_bounded(&chunk_done[mm % NS], static_cast<uint32_t>(mm / NS) & 1u,
                                                     p.dev.err, p.timeout_ns))) {
                set_error(p.dev.err, EP_ERR_TIMEOUT);
                return;
            }
            if (!post_chunk(p, slot_of(mm), nd, gs, ctot, cbb)) return;
        }
        build_meta(p, k, slot_of(m), rbase);
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_full[m % NS]);
    }
    for (int mm = max(0, n_my - NS); mm < n_my; ++mm) {
        if (!__all_sync(kFull, mbar_wait_bounded(&chunk_done[mm % NS], static_cast<uint32_t>(mm / NS) & 1u,
                                                 p.dev.err, p.timeout_ns))) {
            set_error(p.dev.err, EP_ERR_TIMEOUT);
            return;
        }
        if (!post_chunk(p, slot_of(mm), nd, gs, ctot, cbb)) return;
    }
}

// ------------------------------------------------------------ consumer warp
constexpr int kMaxPollRounds = 16;   // up to 512 slots examined per step

__device__ void consumer_warp(const DispatchParams &p, int c, long long expected) {
    const int lane = threadIdx.x & 31;
    unsigned long long *tail = p.dev.tail + static_cast<int64_t>(c) * kHeadStride;
    const unsigned long long base = ld_relaxed(tail);
    const unsigned long long end = base + static_cast<unsigned long long>(expected);
    // every slot that can be outstanding (max_inflight), polled drain_batch at a time
    int window = max(p.drain_batch, ((p.max_inflight + 31) / 32) * 32);
    window = min(window, 32 * kMaxPollRounds);
    const unsigned long long dmask = static_cast<unsigned long long>(p.D - 1);
    const int64_t ring0 = static_cast<int64_t>(c) * p.D;
    unsigned long long pos = base;
    uint64_t idle_since = globaltimer_ns();
    unsigned sleep = 32;
    while (pos < end) {
        const int avail = static_cast<int>(min(end - pos, static_cast<unsigned long long>(window)));
        const int rounds = (avail + 31) / 32;
        // all status loads of the step in flight together
        bool pub[kMaxPollRounds];
#pragma unroll
        for (int q = 0; q < kMaxPollRounds; ++q) {
            pub[q] = false;
            const int off = q * 32 + lane;
            if (q < rounds && off < avail) {
                const unsigned long long idx = pos + static_cast<unsigned long long>(off);
                pub[q] = ld_acquire(p.dev.status + ring0 + static_cast<int64_t>(idx & dmask)) == 2ull * idx + 1ull;
            }
        }
        // the longest run of published slots from pos
        int ready = 0;
#pragma unroll
        for (int q = 0; q < kMaxPollRounds; ++q) {
            if (q >= rounds || ready < q * 32) break;
            const unsigned bal = __ballot_sync(kFull, pub[q]);
            ready += bal == kFull ? 32 : __ffs(~bal) - 1;
        }
        if (ready > 0) {
#pragma unroll
            for (int q = 0; q < kMaxPollRounds; ++q) {
                const int off = q * 32 + lane;
                if (off < ready) {
                    const unsigned long long idx = pos + static_cast<unsigned long long>(off);
                    const int64_t sidx = ring0 + static_cast<int64_t>(idx & dmask);
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.dev.slots + sidx);
                    uint4 *dst = reinterpret_cast<uint4 *>(p.dev.log + static_cast<int64_t>(c) * p.log_cap +
                                                           static_cast<int64_t>(idx - base));
                    const uint4 a = __ldcg(src), b = __ldcg(src + 1);
                    dst[0] = a;
                    dst[1] = b;
                    st_relaxed(p.dev.status + sidx, 2ull * idx + 2ull);   // COMPLETED
                }
            }
            pos += static_cast<unsigned long long>(ready);
            __syncwarp();
            if (lane == 0) st_release(tail, pos);
            idle_since = globaltimer_ns();
            sleep = 32;
        } else {
            if (read_error(p.dev.err) != 0) break;
            if (globaltimer_ns() - idle_since > p.timeout_ns) {
                set_error(p.dev.err, EP_ERR_TIMEOUT);
                break;
            }
            __nanosleep(sleep);
            sleep = min(sleep * 2u, 256u);
        }
    }
    if (lane == 0) p.dev.log_count[c] = static_cast<int64_t>(pos - base);
}

__global__ void __launch_bounds__(kThreads, 1) dispatch_kernel(const DispatchParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const SmemLayout L(p.R, p.C, p.stage_bytes, p.stages, p.meta_slots);
    int *scratch = reinterpret_cast<int *>(smem + L.scratch_off);
    int *flags = scratch + 3 * p.R + 2 * p.C + 1;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *bar_full = bars, *meta_full = bars + p.stages, *chunk_done = meta_full + p.meta_slots;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Prologue: barriers, window starts, and the checks every CTA takes alike
    // so that either all of them run or none does.
    if (warp == kCopyWarp && lane == 0) {
        for (int i = 0; i < p.stages; ++i) mbar_init(&bar_full[i], 1);
        for (int i = 0; i < p.meta_slots; ++i) {
            mbar_init(&meta_full[i], 1);
            mbar_init(&chunk_done[i], 1);
        }
        mbar_fence_init();
    }
    long long my_expected = 0;
    if (warp == kMetaWarp) {
        for (int d = lane; d < p.R; d += 32) scratch[d] = __ldg(p.recv_base + d);
        // N against the receive capacity; every channel's count against its log
        const long long n_recv = static_cast<long long>(__ldg(p.recv_base + p.R - 1)) + __ldg(p.recv_count + p.R - 1);
        long long worst = 0;
        for (int c = 0; c < p.C; ++c) {
            long long part = 0;
            for (int i = lane; i < p.R * p.R; i += 32)
                if ((i % p.R) % p.C == c) part += __ldg(p.msg_count + i);
            for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
            worst = max(worst, part);
        }
        if (lane == 0) {
            int abort = read_error(p.dev.err) != 0;
            if (n_recv > p.cap_rows || n_recv < 0) {
                set_error(p.dev.err, EP_ERR_CAPACITY);
                abort = 1;
            }
            if (worst > p.log_cap) {
                set_error(p.dev.err, EP_ERR_INVALID_ARG);
                abort = 1;
            }
            flags[0] = abort;
        }
    }
    if (warp == kConsumerWarp && static_cast<int>(blockIdx.x) < p.C) {
        const int c = blockIdx.x;
        long long part = 0;
        for (int i = lane; i < p.R * p.R; i += 32)
            if ((i % p.R) % p.C == c) part += __ldg(p.msg_count + i);
        for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
        my_expected = part;
    }
    __syncthreads();
    if (flags[0]) return;

    if (warp == kCopyWarp) {
        copy_warp(p, smem, L, bar_full, meta_full, chunk_done);
    } else if (warp == kMetaWarp) {
        meta_warp(p, smem, L, meta_full, chunk_done, scratch);
    } else if (static_cast<int>(blockIdx.x) < p.C && !(p.debug & EP_DEBUG_DISABLE_CONSUMER)) {
        consumer_warp(p, blockIdx.x, my_expected);
    }
}

}  // namespace

// Geometry: one CTA per SM; stages sized so that a stage holds a run of whole
// rows (rows <= 16 KB) or one piece of a row, and as many stages as fit.
ep_status plan_dispatch(ep_ctx *h) {
    const int R = h->cfg.num_ranks, C = h->cfg.channels;
    const int64_t B = 2ll * h->cfg.hidden;
    const int kTargetStage = 16384;
    int rows_per_item = 1, pieces = 1, piece_bytes = static_cast<int>(B);
    if (B <= kTargetStage) {
        rows_per_item = static_cast<int>(kTargetStage / B);
        if (rows_per_item > kChunkTokens) rows_per_item = kChunkTokens;
        piece_bytes = static_cast<int>(B);
    } else {
        pieces = static_cast<int>((B + kTargetStage - 1) / kTargetStage);
        piece_bytes = static_cast<int>(((B + pieces - 1) / pieces + 15) / 16 * 16);
    }
    const int stage_bytes = ((rows_per_item * piece_bytes) + 127) / 128 * 128;
    const int meta_slots = 3;
    int max_smem = 0;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess)
        return EP_ERR_CUDA;
    const int reserve = 1024;   // static + alignment slack
    int stages = 0;
    for (int s = 15; s >= 3; --s) {
        SmemLayout L(R, C, stage_bytes, s, meta_slots);
        if (L.total + reserve <= max_smem) {
            stages = s;
            break;
        }
    }
    if (stages == 0) return EP_ERR_INVALID_ARG;
    SmemLayout L(R, C, stage_bytes, stages, meta_slots);
    h->rows_per_item = rows_per_item;
    h->pieces = pieces;
    h->piece_bytes = piece_bytes;
    h->stage_bytes = stage_bytes;
    h->stages = stages;
    h->prefetch = stages / 2;
    h->meta_slots = meta_slots;
    h->disp_smem = static_cast<size_t>(L.total);
    h->disp_threads = kThreads;
    h->chunks_per_rank = (h->cfg.tokens_per_rank + kChunkTokens - 1) / kChunkTokens;
    h->nchunks = h->chunks_per_rank * R;
    if (cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(h->disp_smem)) != cudaSuccess)
        return EP_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel, kThreads, h->disp_smem) !=
            cudaSuccess ||
        per_sm < 1)
        return EP_ERR_CUDA;
    h->disp_grid = h->sm_count * 1;
    if (h->disp_grid < C) return EP_ERR_INVALID_ARG;
    return EP_OK;
}

ep_status launch_dispatch(ep_ctx *h, const void *x, const ep_layout_out *lay, void *recv, int64_t cap_rows,
                          cudaStream_t st) {
    DispatchParams p{};
    p.x = static_cast<const uint8_t *>(x);
    p.recv = static_cast<uint8_t *>(recv);
    p.cap_rows = cap_rows < INT32_MAX ? cap_rows : INT32_MAX;   // receive rows are int32
    p.token_slot = lay->token_slot;
    p.recv_base = lay->recv_base;
    p.recv_count = lay->recv_count;
    p.recv_off = lay->recv_off;
    p.send_off = lay->send_off;
    p.cnt = lay->num_tokens_per_rank;
    p.msg_count = lay->msg_count;
    p.dev = h->dev;
    p.R = h->cfg.num_ranks;
    p.Tpr = h->cfg.tokens_per_rank;
    p.T = static_cast<int64_t>(p.R) * p.Tpr;
    p.row_bytes = 2ll * h->cfg.hidden;
    p.log_cap = h->log_cap;
    p.timeout_ns = h->cfg.timeout_ns;
    p.C = h->cfg.channels;
    p.D = h->cfg.ring_depth;
    p.max_inflight = h->cfg.max_inflight;
    p.batch = h->cfg.batch;
    p.G = h->G;
    p.drain_batch = h->cfg.drain_batch;
    p.debug = h->cfg.debug_flags;
    p.chunks_per_rank = h->chunks_per_rank;
    p.nchunks = h->nchunks;
    p.rows_per_item = h->rows_per_item;
    p.pieces = h->pieces;
    p.piece_bytes = h->piece_bytes;
    p.stage_bytes = h->stage_bytes;
    p.stages = h->stages;
    p.prefetch = h->prefetch;
    p.meta_slots = h->meta_slots;
    p.msgs_per_pair = h->msgs_per_pair;
    p.slot_vec = (p.R % 4 == 0 && reinterpret_cast<uintptr_t>(lay->token_slot) % 16 == 0) ? 1 : 0;
    void *args[] = {&p};
    const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(dispatch_kernel),
                                                      dim3(h->disp_grid), dim3(kThreads), args, h->disp_smem, st);
    return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace ep
