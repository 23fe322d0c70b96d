// ep_dispatch.cu -- EP dispatch with TransferCmd rings (sm_103a).
//
// What it does (UCCL-EP article: s6 "Dispatch"; s2.2 the lock-free ring of
// TransferCmd records with head/tail atomics, batch enqueue of up to 8
// commands and flow control against kMaxInflight; s2.3 the TransferCmd fields
// {dst_rank, src_offset, dst_offset, size}; s3.1 Write completes when the
// target memory is visible, Drain waits until the queue is empty; s4.1 the
// pipelined DispatchKernel -- prepare, then post, then go on -- and packing of
// small tokens; s4.2 independent channels; NCCL GIN article s2.2.1 byte-offset
// windows):
//
//   for every token t and destination rank d with token_slot[t][d] >= 0:
//       recv[recv_base[d] + token_slot[t][d]] <- x[t]        (one copy per rank)
//   for every message g of pair (s, d) -- up to G consecutive rows of the pair --
//       post TransferCmd{d, rows*B, (send_off[s][d] + gG)*B, (recv_off[s][d] + gG)*B}
//       into ring d % C once all its rows have landed.
//
// How: one persistent cooperative kernel, one CTA per SM, in two kinds.
//
// Copy CTAs (all but the first C) move the rows.  Chunks of 4 to 32 tokens of
// one source rank (about four per copy CTA at least) are drawn from a
// device-wide counter (so faster SMs take more);
// their warps hand each chunk on through mbarriers and shared counters:
//   copy    1-D TMA bulk loads of token rows (a run of whole rows when they
//           are small, a piece of one row when it is large) into a ring of
//           shared-memory stages, then one TMA bulk store per (row,
//           destination) from the stage; each source row is read from HBM
//           once whatever its number of destinations.  Lane 0 issues the
//           loads; all 32 lanes issue stores, each tracking its own bulk
//           groups, so a stage is recycled only once every lane's stores from
//           it have completed.
//   store   (rows of at most 4 KB only) seven warps take the stores over:
//           the copy warp only loads, and the store warps move each (row,
//           destination) pair from the stage with 16-byte vector stores --
//           a TMA bulk store costs about the same whatever its size, so for
//           small rows TMA, not HBM, would set the pace.
//   meta    reads the chunk's token_slot rows; builds each token's
//           destination-row list (for the copy warp) and writes the chunk's
//           notice -- the first and last window slot it covers per
//           destination rank -- to global memory.
//   notify  once the chunk's stores are complete, fences and sets the
//           chunk's ready flag (tagged with the dispatch's generation).
//
// Channel CTAs (the first C) each own ring c = blockIdx.x:
//   poster  (eight warps) takes groups of 32 chunks in turn, waits for their
//           ready flags, and turns their notices into the messages of ring c
//           that the chunks complete: a message of G rows is complete in the
//           chunk that holds its last row, since all earlier rows of the pair
//           are in earlier chunks.  It posts them in batches of up to `batch`
//           commands: one atomicAdd on head per batch, a wait while the ring
//           would hold more than max_inflight commands, then the slot stores;
//           then it adds the group's messages to the destinations' arrival
//           signals.
//   poller  examines every slot that can be outstanding (drain_batch = 32 per
//           warp-wide load), takes the longest run of published slots, stages
//           the records for the logger and moves the tail (the retire point)
//           -- the posters read it in shared memory, so flow control costs no
//           round trip.
//   logger  decodes the staged records into TransferCmds, appends them to the
//           channel's log in device memory and publishes the cumulative tail
//           and head there (a command is complete once tail has passed it).
//   The channel finishes when its message count (from msg_count) has been
//   retired: the drain.
//
// A ring lives in its channel CTA's shared memory -- the CTA's posters and
// consumer are its only users -- as self-validating 16-byte records (see
// lap_tag): posting a command is one store, reading it needs no fence, and a
// turn of the ring costs no L2 round trip (which takes microseconds while the
// copy CTAs saturate HBM).  The cumulative head and tail the host reads, and
// the logs, are in device memory.  The copy path never waits on a ring.
// Every wait is bounded by the handle's timeout and by the grid's error word;
// none traps.  A cooperative launch keeps every CTA resident while others
// wait on it.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kThreads = 320;   // channel CTAs use all ten warps; copy CTAs three, or ten for small rows
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMetaSlots = 3;       // destination lists in flight (copy CTAs)
constexpr int kDoneSlots = 32;      // chunks stored but not yet reported complete
constexpr int kPrefetchItems = 4;   // row loads in flight per copy CTA
constexpr int kStoreLagItems = 2;   // items whose stores may still be in flight
constexpr int kMaxPollRounds = 16;  // up to 512 slots examined per consumer step
constexpr int kLogStage = 1024;     // staged records (16 bytes each) awaiting the logger
constexpr uint64_t kErrCheckNs = 20000;   // idle loops read the device error word this often
constexpr int kPosterWarpsMax = 8;        // poster warps of a channel CTA, at most
constexpr int kListPerLane = 8;           // commands a poster lane lists per posting pass
constexpr int kMetaLoads = 8;             // int4 token_slot loads a meta lane keeps in flight
constexpr int kNoticeLoads = 8;           // notice entries a poster lane keeps in flight

// Shared words (u64) after rbase: abort flag; chunks complete (copy CTA) or
// ring tail = retire point (channel CTA); poller stopped; ring base; dispatch
// generation; messages expected on the channel; ring head; records logged;
// chunk ids drawn (copy CTA); chunks stored in all, once known (copy CTA);
// items loaded in all + 1, once known (copy CTA, vector-store path); chunks
// flagged by the notify warp (copy CTA); message counters in shared memory
// + 1, or 0 when they live in device memory (channel CTA, G > 1).
// Then, in copy CTAs, the drawn chunk ids (a ring of kIdSlots ints) and, per
// stage, the description of the item it holds (vector-store path).
enum {
    kWAbort = 0, kWProgress = 1, kWStopped = 2, kWBase = 3, kWGen = 4, kWExpected = 5, kWHead = 6, kWLogged = 7,
    kWIds = 8, kWCopyDone = 9, kWItems = 10, kWNotified = 11, kWCounters = 12
};
constexpr int kNumWords = 13;
constexpr int kIdSlots = 32;   // chunk ids a copy CTA has drawn but not yet retired
constexpr int kStagesMax = 15;
constexpr int kSmallPerCta = 6;   // small chunks per copy CTA at the end of a layer

// Rows of at most kVecRowMax bytes leave shared memory by vector stores from
// the copy CTA's store warps (warps kStoreWarp0..) instead of TMA bulk
// stores: a bulk store costs about the same whatever its size, so for small
// rows the TMA unit, not HBM, set the pace.
constexpr int kVecRowMax = 4096;
constexpr int kStoreWarp0 = 3;

// Shared-memory carve, identical on host and device.
struct SmemLayout {
    int stage_off, meta_off, meta_slot_bytes, scratch_off, info_off, chan_off, bar_off, total;
    __host__ __device__ static int ring_off(int R) { return ((12 * R * R) + 127) / 128 * 128; }
    // poster ranges: per poster warp, 32 chunks x ceil(R/C) int2
    __host__ __device__ static int ranges_off(int R, int D) { return ring_off(R) + 16 * D + 16 * kLogStage; }
    __host__ __device__ static int ranges_bytes_per_warp(int R, int C) { return 32 * ((R + C - 1) / C) * 8; }
    // poster lists: per poster warp, 32 x kListPerLane packed commands
    __host__ __device__ static int lists_off(int R, int C, int D, int npw) {
        return (ranges_off(R, D) + npw * ranges_bytes_per_warp(R, C) + 15) & ~15;
    }
    static constexpr int kListBytesPerWarp = 32 * kListPerLane * 16;
    // message counters (G > 1): per (source, destination of the ring) the
    // first counter of the pair's messages, then one 16-bit counter per
    // message; in the space below scratch_off that copy CTAs give to stages
    // and meta slots, at least kCounterBytes of it
    __host__ __device__ static int counters_off(int R, int C, int D, int npw) {
        return (lists_off(R, C, D, npw) + npw * kListBytesPerWarp + 15) & ~15;
    }
    static constexpr int kCounterBytes = 32768;
    // npw: the poster warps that run (fewer when their ranges would not fit
    // beside the ring, e.g. 64 destinations on one channel); G: rows per message
    __host__ __device__ SmemLayout(int R, int C, int D, int stage_bytes, int stages, int npw, int G) {
        stage_off = 0;
        // channel CTAs keep the pair tables (3 x R x R ints) and their ring
        // (D slots of 16 bytes) where copy CTAs keep their stages
        const int stage_area = stage_bytes * stages,
                  channel = counters_off(R, C, D, npw) + (G > 1 ? kCounterBytes : 0);
        meta_off = stage_area > channel ? stage_area : channel;
        meta_slot_bytes = ((32 * R + 33) + 3) / 4 * 16;   // dst[32*R] | pref[33]
        scratch_off = meta_off + meta_slot_bytes * kMetaSlots;
        // scratch: rbase[R] ints, kNumWords u64 words, kIdSlots ints,
        // kStagesMax item descriptions (int4)
        info_off = (scratch_off + ((R + 3) & ~3) * 4 + 8 * kNumWords + 4 * kIdSlots + 15) & ~15;
        chan_off = info_off + 16 * kStagesMax;          // per-channel message counts (prologue)
        bar_off = chan_off + 4 * kMaxChannels;
        // barriers: stage_full[stages], meta_full[3], meta_free[3], stage_empty[stages]
        total = bar_off + 8 * (2 * stages + 2 * kMetaSlots);
    }
};

struct MetaSlot {
    int *dst, *pref;
    __device__ MetaSlot(uint8_t *base, int R) {
        dst = reinterpret_cast<int *>(base);
        pref = dst + 32 * R;
    }
};


// Chunk geometry (see DispatchParams): source rank, first token and tokens
// of chunk k; the chunk before it in its rank's token order (or -1); and the
// call's u-th chunk in draw order.
__device__ __forceinline__ int chunk_src(const DispatchParams &p, int k) {
    const int rb = p.R * p.nbig;
    return k < rb ? k / p.nbig : (k - rb) / p.nsmall;
}
__device__ __forceinline__ int64_t chunk_tok0(const DispatchParams &p, int k) {
    const int rb = p.R * p.nbig;
    if (k < rb) {
        const int s = k / p.nbig, i = k - s * p.nbig;
        return static_cast<int64_t>(s) * p.Tpr + static_cast<int64_t>(i) * p.chunk_tokens;
    }
    const int k2 = k - rb, s = k2 / p.nsmall, j = k2 - s * p.nsmall;
    return static_cast<int64_t>(s) * p.Tpr + static_cast<int64_t>(p.nbig) * p.chunk_tokens +
           static_cast<int64_t>(j) * p.small_tokens;
}
__device__ __forceinline__ int chunk_ntok(const DispatchParams &p, int k) {
    const int rb = p.R * p.nbig;
    if (k < rb) return p.chunk_tokens;
    const int j = (k - rb) % p.nsmall;
    return min(p.small_tokens, p.Tpr - p.nbig * p.chunk_tokens - j * p.small_tokens);
}
__device__ __forceinline__ int chunk_pred(const DispatchParams &p, int k) {
    const int rb = p.R * p.nbig;
    if (k < rb) return k % p.nbig != 0 ? k - 1 : -1;
    const int k2 = k - rb, s = k2 / p.nsmall, j = k2 - s * p.nsmall;
    return j != 0 ? k - 1 : (p.nbig > 0 ? s * p.nbig + p.nbig - 1 : -1);
}
__device__ __forceinline__ int call_chunk(const DispatchParams &p, int u) {
    const int nb_call = (p.s1 - p.s0) * p.nbig;
    return u < nb_call ? p.s0 * p.nbig + u : p.R * p.nbig + p.s0 * p.nsmall + (u - nb_call);
}
__device__ __forceinline__ int chunk_items(const DispatchParams &p, int ntok) {
    return p.pieces > 1 ? ntok * p.pieces : (ntok + p.rows_per_item - 1) / p.rows_per_item;
}
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const DispatchParams &p) {
    return __all_sync(kFull, mbar_wait_bounded(bar, parity, p.dev.err, p.timeout_ns));
}

// Walks the items of one chunk: a run of whole rows when they are small, a
// piece of one row when it is large.  k < 0 marks the end of the chunks.
struct ItemCursor {
    int k, q, ntok, nitems;
    __device__ void set_chunk(const DispatchParams &p, int k_) {
        k = k_;
        q = 0;
        ntok = nitems = 0;
        if (k >= 0) {
            ntok = chunk_ntok(p, k);
            nitems = chunk_items(p, ntok);
        }
    }
    __device__ bool valid() const { return k >= 0; }
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

struct Bars {
    uint64_t *stage_full, *meta_full, *meta_free, *stage_empty;
};

// The chunks a copy CTA copies, in order: its first is fixed (copy CTA i
// takes the call's chunk i in draw order), the rest come from a device-wide
// counter, so
// that CTAs on faster SMs take more and all finish together.  Each draw
// publishes the chunk id to the CTA's other warps first and only then asks
// the counter for the next one, so that the atomic's round trip overlaps a
// whole chunk of copying instead of delaying the release.  Warp-uniform.
struct ChunkDraw {
    const DispatchParams &p;
    unsigned long long *words;
    int *ids;
    unsigned int ahead;   // lane 0: index (within the call) of the next chunk
    int n_drawn = 0;
    __device__ ChunkDraw(const DispatchParams &p_, unsigned long long *w, int *i)
        : p(p_), words(w), ids(i), ahead(blockIdx.x - static_cast<unsigned>(p_.C)) {}
    __device__ int next() {
        const int lane = threadIdx.x & 31;
        const unsigned ncopy = gridDim.x - static_cast<unsigned>(p.C);
        int k = -1;
        if (lane == 0) {
            // the ring of ids holds kIdSlots chunks: wait until the notify
            // warp is done with the one this draw replaces
            if (n_drawn >= kIdSlots) {
                const uint64_t t0 = globaltimer_ns();
                ErrPoll ep(t0);
                while (ld_acquire_cta_shared(&words[kWNotified]) <= static_cast<unsigned long long>(n_drawn - kIdSlots)) {
                    const uint64_t tn = globaltimer_ns();
                    if (ep.raised(p.dev.err, tn) || tn - t0 > p.timeout_ns) {
                        if (read_error(p.dev.err) == 0) set_error(p.dev.err, EP_ERR_TIMEOUT);
                        ahead = static_cast<unsigned>(p.nk);   // draw nothing more
                        break;
                    }
                    __nanosleep(64);
                }
            }
            k = ahead < static_cast<unsigned>(p.nk) ? call_chunk(p, static_cast<int>(ahead)) : -1;
            ids[n_drawn % kIdSlots] = k;
        }
        k = __shfl_sync(kFull, k, 0);
        ++n_drawn;
        __syncwarp();
        if (lane == 0) {
            st_release_cta_shared(&words[kWIds], static_cast<unsigned long long>(n_drawn));
            if (k >= 0) ahead = ncopy + atomicAdd(p.dev.chunk_next, 1u);
        }
        return k;
    }
};

// ------------------------------------------------------------ copy CTA: copy
// Chunks are drawn from a device-wide counter as the loads reach them, so
// that CTAs on faster SMs take more chunks and all finish together; the ids
// go to a shared ring for the meta and notify warps.
__device__ void copy_warp(const DispatchParams &p, uint8_t *smem, const SmemLayout &L, const Bars &bars,
                          unsigned long long *words, int *ids) {
    const int lane = threadIdx.x & 31;
    const int S = p.stages, P = p.prefetch;
    const int64_t B = p.row_bytes;
    int64_t n_loaded = 0, n_stored = 0;
    int stored_chunks = 0, reported = 0;
    int64_t last_item[kDoneSlots];   // last item of chunks stored but not yet reported
#pragma unroll
    for (int i = 0; i < kDoneSlots; ++i) last_item[i] = 0;
    bool ok = true;

    ChunkDraw dr(p, words, ids);
    auto draw = [&]() -> int { return dr.next(); };
    ItemCursor ld, stc;
    int ld_m = 0, st_m = 0;
    ld.set_chunk(p, draw());
    stc.set_chunk(p, ld.k);
    auto advance_ld = [&]() {
        if (++ld.q < ld.nitems) return;
        ++ld_m;
        ld.set_chunk(p, draw());
    };
    auto advance_st = [&]() {
        if (++stc.q < stc.nitems) return;
        ++st_m;
        stc.set_chunk(p, ids[st_m % kIdSlots]);   // drawn already: the loads run ahead
    };

    auto issue_load = [&](const ItemCursor &c, int64_t idx) {
        if (lane == 0) {
            int ta, tb, off, len;
            c.geometry(p, ta, tb, off, len);
            const int stage = static_cast<int>(idx % S);
            const uint32_t bytes = static_cast<uint32_t>((tb - ta) * len);
            const uint8_t *src = p.x + (chunk_tok0(p, c.k) + ta) * B + off;
            mbar_arrive_expect_tx(&bars.stage_full[stage], bytes);
            bulk_g2s(smem + L.stage_off + static_cast<int64_t>(stage) * p.stage_bytes, src, bytes,
                     &bars.stage_full[stage]);
        }
    };
    // Report every stored chunk whose last item is <= upto as complete (the
    // notify warp reads the count).
    auto report_upto = [&](int64_t upto) {
        const int before = reported;
        while (reported < stored_chunks && last_item[reported % kDoneSlots] <= upto) ++reported;
        if (reported != before) {
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) st_release_cta_shared(&words[kWProgress], static_cast<unsigned long long>(reported));
        }
    };

    for (int i = 0; i < P && ld.valid(); ++i) {
        issue_load(ld, n_loaded++);
        advance_ld();
    }
    while (stc.valid()) {
        const int64_t i = n_stored;
        const int slot = st_m % kMetaSlots;
        if (stc.q == 0) {
            const uint32_t par = static_cast<uint32_t>(st_m / kMetaSlots) & 1u;
            if (!__all_sync(kFull, mbar_test(&bars.meta_full[slot], par))) {
                // report what has landed before waiting on the meta warp
                bulk_wait<0>();
                report_upto(INT64_MAX);
                if (!warp_wait(&bars.meta_full[slot], par, p)) {
                    set_error(p.dev.err, EP_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
        const int stage = static_cast<int>(i % S);
        if (!warp_wait(&bars.stage_full[stage], static_cast<uint32_t>(i / S) & 1u, p)) {
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
            // every store of the chunk is issued: its destination list is free
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.meta_free[slot]);
            last_item[st_m % kDoneSlots] = i;
            ++stored_chunks;
        }
        ++n_stored;
        advance_st();
        // At most store_lag items' stores stay in flight; the stage of item
        // n_loaded was last used by item n_loaded - S, complete because
        // store_lag <= S - P.
        bulk_wait_n(p.store_lag);
        report_upto(n_stored - 1 - p.store_lag);
        if (ld.valid()) {
            issue_load(ld, n_loaded++);
            advance_ld();
        }
    }
    bulk_wait<0>();
    if (ok) {
        report_upto(INT64_MAX);
    } else {
        // abort: let every load already issued land before the CTA exits (the
        // wait ignores the error word; it is still bounded by the time limit)
        for (int64_t j = n_stored; j < n_loaded; ++j)
            mbar_wait_bounded(&bars.stage_full[j % S], static_cast<uint32_t>(j / S) & 1u, nullptr, p.timeout_ns);
        __syncwarp();
    }
    // the id drawn ahead (if any) is simply unused: the counter only has to
    // be reset between calls, which the last CTA does
    if (lane == 0) st_release_cta_shared(&words[kWCopyDone], ok ? static_cast<unsigned long long>(stored_chunks) + 1ull
                                                                : 1ull);
}

// ------------------------------------------- copy CTA: small rows, loads
// The vector-store path.  The copy warp only loads: per item it waits until
// the item's stage is given back, writes the item's description (meta slot,
// chunk number, tokens, last-of-chunk), and issues the TMA load.  It gives the
// chunk to the notify warp once the store warps have given back every item
// of the chunk (their mbarrier arrivals order their stores before it).
__device__ void copy_warp_vec(const DispatchParams &p, uint8_t *smem, const SmemLayout &L, const Bars &bars,
                              unsigned long long *words, int *ids, int4 *info) {
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int64_t B = p.row_bytes;
    int64_t n_loaded = 0, n_back = 0;
    int chunks = 0, reported = 0;
    int64_t last_item[kDoneSlots];   // last item of chunks loaded but not yet reported
#pragma unroll
    for (int i = 0; i < kDoneSlots; ++i) last_item[i] = 0;
    bool ok = true;

    ChunkDraw dr(p, words, ids);
    auto draw = [&]() -> int { return dr.next(); };
    // take back the items the store warps have finished, in order; report the
    // chunks whose every item is back.  Blocking: wait until item `until` is.
    auto take_back = [&](int64_t until) {
        while (n_back < n_loaded && ok) {
            uint64_t *bar = &bars.stage_empty[n_back % S];
            const uint32_t par = static_cast<uint32_t>(n_back / S) & 1u;
            if (!__all_sync(kFull, mbar_test(bar, par))) {
                if (n_back > until) break;
                if (!warp_wait(bar, par, p)) {
                    set_error(p.dev.err, EP_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
            ++n_back;
        }
        const int before = reported;
        while (reported < chunks && last_item[reported % kDoneSlots] < n_back) ++reported;
        if (reported != before) {
            __syncwarp();
            if (lane == 0) st_release_cta_shared(&words[kWProgress], static_cast<unsigned long long>(reported));
        }
    };

    ItemCursor ld;
    int ld_m = 0;
    ld.set_chunk(p, draw());
    while (ld.valid() && ok) {
        if (n_loaded >= S) take_back(n_loaded - S);   // the stage's previous item
        if (!ok) break;
        fence_proxy_async_shared();   // the store warps' reads of the stage before the refill
        int ta, tb, off, len;
        ld.geometry(p, ta, tb, off, len);
        const int st = static_cast<int>(n_loaded % S);
        const int last = ld.q == ld.nitems - 1;
        if (lane == 0) {
            info[st] = make_int4(ld_m, ta, tb, last);
            const uint32_t bytes = static_cast<uint32_t>((tb - ta) * len);
            const uint8_t *src = p.x + (chunk_tok0(p, ld.k) + ta) * B + off;
            mbar_arrive_expect_tx(&bars.stage_full[st], bytes);   // releases the description too
            bulk_g2s(smem + L.stage_off + static_cast<int64_t>(st) * p.stage_bytes, src, bytes,
                     &bars.stage_full[st]);
        }
        if (last) {
            last_item[chunks % kDoneSlots] = n_loaded;
            ++chunks;
        }
        ++n_loaded;
        if (++ld.q >= ld.nitems) {
            ++ld_m;
            ld.set_chunk(p, draw());
        }
        take_back(-1);
    }
    __syncwarp();
    if (lane == 0) st_release_cta_shared(&words[kWItems], static_cast<unsigned long long>(n_loaded) + 1ull);
    if (ok) {
        take_back(n_loaded - 1);
    } else {
        // abort: let every load already issued land before the CTA exits
        for (int64_t j = n_back; j < n_loaded; ++j)
            mbar_wait_bounded(&bars.stage_full[j % S], static_cast<uint32_t>(j / S) & 1u, nullptr, p.timeout_ns);
        __syncwarp();
    }
    if (lane == 0) st_release_cta_shared(&words[kWCopyDone], ok ? static_cast<unsigned long long>(chunks) + 1ull
                                                                : 1ull);
}

// ------------------------------------------ copy CTA: small rows, stores
// Store warp w of the vector-store path takes, of every item, the (row,
// destination) pairs w, w + store_warps, ...: the 32 lanes move the row from
// the stage to its receive row with 16-byte loads and stores.  Then it gives
// the stage back, and, after the last item of a chunk, the chunk's meta slot.
__device__ void store_warp(const DispatchParams &p, uint8_t *smem, const SmemLayout &L, const Bars &bars,
                           unsigned long long *words, const int4 *info, int w) {
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int64_t B = p.row_bytes;
    const int nseg = static_cast<int>(B / 16);
    int cur_m = -1;
    for (int64_t i = 0;; ++i) {
        const int st = static_cast<int>(i % S);
        const uint32_t par = static_cast<uint32_t>(i / S) & 1u;
        // item i, once loaded, or the end
        const uint64_t t0 = globaltimer_ns();
        ErrPoll ep(t0);
        bool have = false, end = false;
        unsigned nap = 32;
        while (true) {
            have = __all_sync(kFull, mbar_test(&bars.stage_full[st], par));
            if (have) break;
            const unsigned long long items = ld_acquire_cta_shared(&words[kWItems]);
            if (items != 0ull && static_cast<unsigned long long>(i) + 1ull >= items) {
                end = true;
                break;
            }
            const uint64_t now = globaltimer_ns();
            bool give_up = (lane == 0 && ep.raised(p.dev.err, now)) || now - t0 > p.timeout_ns;
            if (__any_sync(kFull, give_up)) {
                if (read_error(p.dev.err) == 0) set_error(p.dev.err, EP_ERR_TIMEOUT);
                end = true;
                break;
            }
            __nanosleep(nap);
            nap = min(nap * 2u, 256u);
        }
        if (end) return;
        const int4 it = info[st];   // m, ta, tb, last
        const int slot = it.x % kMetaSlots;
        if (it.x != cur_m) {
            if (!warp_wait(&bars.meta_full[slot], static_cast<uint32_t>(it.x / kMetaSlots) & 1u, p)) {
                set_error(p.dev.err, EP_ERR_TIMEOUT);
                return;
            }
            cur_m = it.x;
        }
        const MetaSlot ms(smem + L.meta_off + static_cast<int64_t>(slot) * L.meta_slot_bytes, p.R);
        const uint8_t *stage_base = smem + L.stage_off + static_cast<int64_t>(st) * p.stage_bytes;
        const int ta = it.y, tb = it.z;
        const int pb = ms.pref[ta], pe = ms.pref[tb];
        int tl = ta;
        for (int pi = pb + w; pi < pe; pi += p.store_warps) {
            while (ms.pref[tl + 1] <= pi) ++tl;
            const int row = ms.dst[tl * p.R + (pi - ms.pref[tl])];
            const uint8_t *src = stage_base + static_cast<int64_t>(tl - ta) * B;
            uint8_t *dst = p.recv + static_cast<int64_t>(row) * B;
            uint4 v[kVecRowMax / 16 / 32];
#pragma unroll
            for (int q = 0; q < kVecRowMax / 16 / 32; ++q)
                if (lane + 32 * q < nseg) v[q] = ld_shared_v4(src + 16 * (lane + 32 * q));
#pragma unroll
            for (int q = 0; q < kVecRowMax / 16 / 32; ++q)
                if (lane + 32 * q < nseg) *reinterpret_cast<uint4 *>(dst + 16 * (lane + 32 * q)) = v[q];
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bars.stage_empty[st]);
            if (it.w) mbar_arrive(&bars.meta_free[slot]);
        }
    }
}

// ------------------------------------------------------------ copy CTA: meta
__device__ void build_meta_by_token(const DispatchParams &p, int k, const MetaSlot &ms, const int *rbase) {
    const int lane = threadIdx.x & 31;
    const int R = p.R;
    const int ntok = chunk_ntok(p, k);
    const int64_t tok0 = chunk_tok0(p, k);
    const bool valid = lane < ntok;
    const int64_t t = tok0 + lane;
    int32_t *notice = p.dev.notice + static_cast<int64_t>(k) * 2 * R;
    int n = 0;
    int *dst = ms.dst + lane * R;
    // lane = token.  Its token_slot row, kMetaLoads x 4 destinations per
    // batch: every load of a batch is issued before any is used, so a batch
    // costs one memory round trip; then, per destination, the lane appends
    // the receive row to its own list and two warp reductions give the
    // chunk's first and last window slot (the notice)
    for (int d00 = 0; d00 < R; d00 += 4 * kMetaLoads) {
        int4 q[kMetaLoads];
#pragma unroll
        for (int b = 0; b < kMetaLoads; ++b) {
            const int d0 = d00 + 4 * b;
            q[b] = make_int4(-1, -1, -1, -1);
            if (valid && d0 < R) {
                if (p.slot_vec) {
                    q[b] = __ldg(reinterpret_cast<const int4 *>(p.token_slot + t * R + d0));
                } else {
                    if (d0 + 0 < R) q[b].x = __ldg(p.token_slot + t * R + d0 + 0);
                    if (d0 + 1 < R) q[b].y = __ldg(p.token_slot + t * R + d0 + 1);
                    if (d0 + 2 < R) q[b].z = __ldg(p.token_slot + t * R + d0 + 2);
                    if (d0 + 3 < R) q[b].w = __ldg(p.token_slot + t * R + d0 + 3);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kMetaLoads; ++b) {
            const int d0 = d00 + 4 * b;
            if (d0 >= R) break;
            const int v[4] = {q[b].x, q[b].y, q[b].z, q[b].w};
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
                if (lane == (d & 31)) {
                    notice[2 * d] = lo == INT32_MAX ? -1 : lo;
                    notice[2 * d + 1] = hi;
                }
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
}

__device__ void build_meta_by_dest(const DispatchParams &p, int k, const MetaSlot &ms, const int *rbase) {
    const int lane = threadIdx.x & 31;
    const int R = p.R;
    const int ntok = chunk_ntok(p, k);
    const int64_t tok0 = chunk_tok0(p, k);
    int32_t *notice = p.dev.notice + static_cast<int64_t>(k) * 2 * R;
    int *buf = ms.dst;   // [32 x R]: the chunk's token_slot rows, then each token's receive rows
    // 1. lane = token: its token_slot row (kMetaLoads x 4 destinations per
    //    batch, every load of a batch issued before the first is stored)
    {
        const bool valid = lane < ntok;
        const int64_t t = tok0 + lane;
        int *row = buf + lane * R;
        for (int d00 = 0; d00 < R; d00 += 4 * kMetaLoads) {
            int4 q[kMetaLoads];
#pragma unroll
            for (int b = 0; b < kMetaLoads; ++b) {
                const int d0 = d00 + 4 * b;
                q[b] = make_int4(-1, -1, -1, -1);
                if (valid && d0 < R) {
                    if (p.slot_vec) {
                        q[b] = __ldg(reinterpret_cast<const int4 *>(p.token_slot + t * R + d0));
                    } else {
                        if (d0 + 0 < R) q[b].x = __ldg(p.token_slot + t * R + d0 + 0);
                        if (d0 + 1 < R) q[b].y = __ldg(p.token_slot + t * R + d0 + 1);
                        if (d0 + 2 < R) q[b].z = __ldg(p.token_slot + t * R + d0 + 2);
                        if (d0 + 3 < R) q[b].w = __ldg(p.token_slot + t * R + d0 + 3);
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < kMetaLoads; ++b) {
                const int d0 = d00 + 4 * b;
                if (d0 + 0 < R) row[d0 + 0] = q[b].x;
                if (d0 + 1 < R) row[d0 + 1] = q[b].y;
                if (d0 + 2 < R) row[d0 + 2] = q[b].z;
                if (d0 + 3 < R) row[d0 + 3] = q[b].w;
            }
        }
    }
    __syncwarp();
    // 2. lane = destination: per token, one ballot places the destination in
    //    the token's list (token j's rows in increasing destination order,
    //    written over its staged slots: a row lands at or before the slot it
    //    came from, after every lane has read that slot); lane j keeps token
    //    j's count.  The first and last window slots of the chunk per
    //    destination are the notice.
    const unsigned lt = (1u << lane) - 1u;
    int mine = 0;   // lane j: receive rows listed for token j
    for (int g = 0; g * 32 < R; ++g) {
        const int d = g * 32 + lane;
        const bool dv = d < R;
        const int64_t rb = dv ? rbase[d] : 0;
        int lo = -1, hi = -1;
#pragma unroll 4
        for (int j = 0; j < ntok; ++j) {
            const int v = dv ? buf[j * R + d] : -1;
            const bool member = v >= 0;
            const unsigned bal = __ballot_sync(kFull, member);
            const int cj = g > 0 ? __shfl_sync(kFull, mine, j) : 0;
            if (member) {
                const int64_t r = rb + v;
                if (r >= 0 && r < p.cap_rows) {
                    buf[j * R + cj + __popc(bal & lt)] = static_cast<int>(r);
                } else {
                    set_error(p.dev.err, EP_ERR_CAPACITY);
                }
                if (lo < 0) lo = v;
                hi = v;
            }
            if (lane == j) mine += __popc(bal);
        }
        if (dv) *reinterpret_cast<int2 *>(notice + 2 * d) = make_int2(lo, hi);
    }
    // 3. list starts: exclusive prefix of the tokens' list lengths
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    ms.pref[lane] = incl - mine;
    if (lane == 31) ms.pref[32] = incl;
}

// The chunk's destination lists (MetaSlot: per token, its receive rows in
// increasing destination order; pref: where each token's list starts in the
// chunk's sequence of (row, destination) pairs) and its notice (the first
// and last window slot per destination rank).  Two equivalent builders: by
// destination for chunks of up to 8 tokens -- a few ballots, and short, which
// matters because the first chunk's lists hold up every copy CTA's first
// stores -- and by token for larger chunks, where it measured faster.
__device__ void build_meta(const DispatchParams &p, int k, const MetaSlot &ms, const int *rbase) {
    if (chunk_ntok(p, k) <= 8)
        build_meta_by_dest(p, k, ms, rbase);
    else
        build_meta_by_token(p, k, ms, rbase);
}

__device__ void meta_warp(const DispatchParams &p, uint8_t *smem, const SmemLayout &L, const Bars &bars,
                          const int *rbase, unsigned long long *words, const int *ids) {
    const int lane = threadIdx.x & 31;
    for (int m = 0;; ++m) {
        // chunk id m, once the copy warp has drawn it
        const uint64_t t0 = globaltimer_ns();
        ErrPoll ep(t0);
        bool ok = true;
        while (ld_acquire_cta_shared(&words[kWIds]) <= static_cast<unsigned long long>(m)) {
            const uint64_t now = globaltimer_ns();
            if (ep.raised(p.dev.err, now) || now - t0 > p.timeout_ns) {
                ok = false;
                break;
            }
            __nanosleep(64);
        }
        if (!__all_sync(kFull, ok)) {
            set_error(p.dev.err, EP_ERR_TIMEOUT);
            return;
        }
        const int k = ids[m % kIdSlots];
        if (k < 0) return;
        if (m >= kMetaSlots &&
            !warp_wait(&bars.meta_free[m % kMetaSlots], static_cast<uint32_t>(m / kMetaSlots - 1) & 1u, p)) {
            set_error(p.dev.err, EP_ERR_TIMEOUT);
            return;
        }
        build_meta(p, k, MetaSlot(smem + L.meta_off + static_cast<int64_t>(m % kMetaSlots) * L.meta_slot_bytes, p.R),
                   rbase);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.meta_full[m % kMetaSlots]);
    }
}

// ---------------------------------------------------------- copy CTA: notify
// Sets ready[k] once chunk k's rows are complete: the copy warp counts
// completed chunks in shared memory; one gpu-scope fence covers every chunk
// reported since the last one.
__device__ void notify_warp(const DispatchParams &p, unsigned long long *words, const int *ids) {
    if ((threadIdx.x & 31) != 0) return;
    const unsigned int tag = static_cast<unsigned int>(words[kWGen]) + 1u;
    int done = 0;
    uint64_t idle_since = globaltimer_ns();
    ErrPoll ep(idle_since);
    unsigned sleep = 32;
    while (true) {
        const int now = static_cast<int>(ld_acquire_cta_shared(&words[kWProgress]));
        if (now > done) {
            fence_acq_rel_gpu();   // the chunks' rows are visible device-wide before their flags
            for (int m = done; m < now; ++m) st_relaxed_u32(p.dev.ready + ids[m % kIdSlots], tag);
            done = now;
            st_release_cta_shared(&words[kWNotified], static_cast<unsigned long long>(done));
            idle_since = globaltimer_ns();
            sleep = 32;
            continue;
        }
        const unsigned long long fin = ld_acquire_cta_shared(&words[kWCopyDone]);
        if (fin != 0ull && static_cast<int>(ld_acquire_cta_shared(&words[kWProgress])) == done) break;
        const uint64_t tnow = globaltimer_ns();
        if (ep.raised(p.dev.err, tnow)) break;
        if (tnow - idle_since > p.timeout_ns) {
            set_error(p.dev.err, EP_ERR_TIMEOUT);
            break;
        }
        __nanosleep(sleep);
        sleep = min(sleep * 2u, 256u);
    }
}

// ------------------------------------------------------ channel CTA: poster

// A ring slot holds one TransferCmd packed into two 64-bit words, each tagged
// with the slot's lap (command index / D) in 16 bits.  Every offset of a
// command is a whole number of rows, so the words carry rows, not bytes:
//   w0 = lap:16 | dst_rank:6 | rows:11 | src_row:31   (src_offset = src_row * B, size = rows * B)
//   w1 = lap:16 | 0:17       | dst_row:31             (dst_offset = dst_row * B)
// A 64-bit access is single-copy atomic, so a consumer that finds both tags
// equal to the lap it expects has the whole record of this lap.
__device__ __forceinline__ unsigned long long lap_tag(unsigned long long idx, int lg_depth) {
    // top bit set, low 15 bits of the lap: consecutive laps of a slot differ
    // and no lap reads as the zeroed slots of a fresh ring
    const unsigned lap = static_cast<unsigned>(idx >> lg_depth);
    return static_cast<unsigned long long>(0x8000u | (lap & 0x7FFFu)) << 48;
}

// Per-lane ring statistics, reduced once at the end of the kernel.
struct LaneStats {
    unsigned long long batches = 0, stalls = 0;
    unsigned max_batch = 0, max_inflight = 0;
};

// Pair tables (num_tokens_per_rank, recv_off, send_off; [R, R] each), staged
// in a channel CTA's shared memory so that turning a notice into commands
// costs no round trip.
struct PairTables {
    const int *cnt, *recv0, *send0;
};

// The messages of pair (s, d) that one chunk's rows [jlo, jhi] of the pair
// touch: g in [ga, gz], message g being rows [gG, min(gG + G, cnt)).  A
// message that also has rows outside the chunk (G > 1) is shared with other
// chunks and posted by whichever of them lands last: each adds the rows it
// holds (rowsa, rowsz) to the message's counter, and the add that brings the
// count to the message's size posts it.
struct MsgSpan {
    int ga, gz, za, zz, enda, endz;
    unsigned rowsa, rowsz;
    bool sha, shz;   // first / last message shared with other chunks
    // lh: the chunk's first and last receive rows for the pair; false when
    // they are not rows of the pair
    __device__ __forceinline__ bool init(int2 lh, int cnt, int r0, int G) {
        const int jlo = lh.x - r0, jhi = lh.y - r0;
        if (jlo < 0 || jhi < jlo || jhi >= cnt) return false;
        ga = jlo / G;
        gz = jhi / G;
        za = ga * G;
        zz = gz * G;
        enda = min(za + G, cnt) - 1;
        endz = min(zz + G, cnt) - 1;
        sha = G > 1 && (za < jlo || (ga == gz && enda > jhi));
        shz = G > 1 && ga != gz && endz > jhi;
        rowsa = static_cast<unsigned>(min(enda, jhi) - max(za, jlo) + 1);
        rowsz = static_cast<unsigned>(jhi - zz + 1);
        return true;
    }
    // messages [gb, ge) this chunk posts, given the counters' values before
    // its adds; fa / fz: its add completed the first / last message
    __device__ __forceinline__ int2 posts(unsigned olda, unsigned oldz, bool &fa, bool &fz) const {
        int gb = ga, ge = gz + 1;
        fa = sha && olda + rowsa == static_cast<unsigned>(enda - za + 1);
        fz = shz && oldz + rowsz == static_cast<unsigned>(endz - zz + 1);
        if (sha && !fa) {
            if (ga == gz)
                ge = gb;
            else
                gb = ga + 1;
        }
        if (shz && !fz) ge = gz;
        return make_int2(gb, ge);
    }
};

// Adds v to 16-bit counter m of a shared-memory array of them (two to a
// word; a count never reaches 2^16) and returns its old value.
__device__ __forceinline__ unsigned add_half_counter(unsigned *ctr, int m, unsigned v) {
    const int sh = (m & 1) * 16;
    return (atom_add_acq_rel_cta_shared(ctr + (m >> 1), v << sh) >> sh) & 0xffffu;
}

// The poster's span pass for counters in device memory (a ring whose
// messages outnumber its shared-memory room): relaxed adds, kNoticeLoads
// destinations' adds in flight at once, bracketed by a release fence before
// them and an acquire fence after a completing one; a completed counter is
// left at zero for the next call.  Writes the chunk's messages to post per
// destination to rg[0, nd) and returns their number, or -1 when a notice
// is out of range.
__device__ __forceinline__ int device_counter_spans(unsigned *msg_rows, PairTables pt, int R, int C, int G, int c, int s,
                                                 int nd, const int32_t *nt, int2 *rg) {
    int total = 0;
    bool bad = false;
    fence_acq_rel_gpu();
    bool done = false;
    for (int i0 = 0; i0 < nd; i0 += kNoticeLoads) {
        int2 lhs[kNoticeLoads];
        unsigned olda[kNoticeLoads], oldz[kNoticeLoads];
#pragma unroll
        for (int b = 0; b < kNoticeLoads; ++b)
            lhs[b] = i0 + b < nd ? __ldcg(reinterpret_cast<const int2 *>(nt + 2 * (c + (i0 + b) * C)))
                                 : make_int2(-1, -1);
#pragma unroll
        for (int b = 0; b < kNoticeLoads; ++b) {
            const int d = c + (i0 + b) * C;
            MsgSpan sp;
            olda[b] = oldz[b] = 0u;
            if (lhs[b].y >= 0 && sp.init(lhs[b], pt.cnt[s * R + d], pt.recv0[s * R + d], G)) {
                unsigned *q = msg_rows + pt.send0[s * R + d];
                if (sp.sha) olda[b] = atom_add_relaxed(q + sp.za, sp.rowsa);
                if (sp.shz) oldz[b] = atom_add_relaxed(q + sp.zz, sp.rowsz);
            }
        }
#pragma unroll
        for (int b = 0; b < kNoticeLoads; ++b) {
            const int i = i0 + b, d = c + i * C;
            if (i >= nd) continue;
            int2 r = make_int2(0, 0);
            MsgSpan sp;
            if (lhs[b].y >= 0 && !sp.init(lhs[b], pt.cnt[s * R + d], pt.recv0[s * R + d], G)) {
                bad = true;
            } else if (lhs[b].y >= 0) {
                bool fa, fz;
                r = sp.posts(olda[b], oldz[b], fa, fz);
                unsigned *q = msg_rows + pt.send0[s * R + d];
                if (fa) q[sp.za] = 0u;
                if (fz) q[sp.zz] = 0u;
                done = done || fa || fz;
            }
            rg[i] = r;
            total += r.y - r.x;
        }
    }
    if (done) fence_acq_rel_gpu();
    return bad ? -1 : total;
}

// The posters of ring c.  Poster warp w takes chunk groups w, w + kPosterWarps,
// ... of 32 chunks, lane i holding chunk 32 * group + i.  It polls the
// group's ready flags and takes, pass by pass, the chunks found ready: each
// such lane loads its chunk's notice for every destination of ring c (one
// round trip) and derives the messages the chunk completes on ring c: those
// of pair (s, d) all of whose rows lie in the chunk's rows [jlo, jhi] of the
// pair, and those it shares with other chunks whose counter its add brings to
// the message's size (MsgSpan).  The ranges go to shared memory.  Then every lane writes its chunk's next commands (packed
// as a slot holds them) into the warp's list -- a walk along its own ranges,
// no search -- and the warp posts the list one command per lane, 32 a round:
// the first lane of each batch of up to `batch` lanes reserves the batch's
// slots with one atomicAdd on head, and each lane stores its slot as soon as
// base + n - tail <= max_inflight (tail is the poller's retire point, in
// shared memory).
constexpr int kPosterWarps = 8;
// Channel-CTA warps: warps 3 and 5 are the poller and the logger; the other
// eight post.
constexpr int kPollWarp = 3, kLogWarp = 5;
static_assert(kThreads / 32 == kPosterWarps + 2, "one warp per poster, plus the poller and the logger");
__device__ __forceinline__ int poster_index(int warp) { return warp - (warp > kPollWarp) - (warp > kLogWarp); }

__device__ void poster_warp(const DispatchParams &p, int c, int w, unsigned long long *words, const PairTables &pt,
                            unsigned long long *ring, int2 *ranges, unsigned long long *list, int *msgoff) {
    const int lane = threadIdx.x & 31;
    const int R = p.R, C = p.C, G = p.G;
    const int nd = c < R ? (R - 1 - c) / C + 1 : 0;   // destinations d = c, c + C, ... on this ring
    // message counters for G > 1: in shared memory when they fit (msgoff
    // gives each pair's first), else in device memory at each message's
    // first send row
    unsigned *ctr_smem = (G > 1 && words[kWCounters] != 0ull) ? reinterpret_cast<unsigned *>(msgoff) + R * nd : nullptr;
    const int ndmax = (R + C - 1) / C;
    const unsigned long long dmask = static_cast<unsigned long long>(p.D - 1);
    const unsigned long long limit = static_cast<unsigned long long>(p.max_inflight);
    const unsigned int tag = static_cast<unsigned int>(words[kWGen]) + 1u;
    unsigned long long *head = &words[kWHead];
    const int rs = 32 - (32 % p.batch);               // commands per round: whole batches
    const int leader = (lane / p.batch) * p.batch;    // first lane of this lane's batch
    LaneStats st;
    bool failed = false;
    const int ngroups = nd > 0 ? (p.nk + 31) / 32 : 0;
    uint64_t err_checked = globaltimer_ns();
    for (int grp = w; grp < ngroups && !failed; grp += p.poster_warps) {
        const int u = grp * 32 + lane;   // this lane's chunk: the call's u-th
        const int k = u < p.nk ? call_chunk(p, u) : -1;
        // Post the group's chunks as they become ready: wait until at least
        // one pending chunk's flag is set (polling device memory with a
        // back-off), post every chunk found ready, and come back for the
        // rest.  While posting, the warp touches shared memory only and
        // answers the ring at once.
        bool pending = u < p.nk;          // this lane's chunk is not yet posted
        const uint64_t tw = globaltimer_ns();
        ErrPoll ep(tw);
        while (__any_sync(kFull, pending) && !failed) {
            bool take_now = false;
            {
                unsigned nap = 128;
                while (true) {
                    if (pending && !take_now) take_now = ld_acquire_u32(p.dev.ready + k) == tag;
                    if (__any_sync(kFull, take_now)) break;
                    const uint64_t now = globaltimer_ns();
                    const bool give_up = (lane == 0 && ep.raised(p.dev.err, now)) || (pending && now - tw > p.timeout_ns);
                    if (__any_sync(kFull, give_up)) {
                        if (read_error(p.dev.err) == 0) set_error(p.dev.err, EP_ERR_TIMEOUT);
                        failed = true;
                        break;
                    }
                    __nanosleep(nap);
                    nap = min(nap * 2u, 2048u);
                }
                if (failed) break;
            }
            pending = pending && !take_now;
            // this lane's chunk: messages [gb, ge) per destination of ring c
            int total = 0;
            if (take_now) {
                const int s = chunk_src(p, k);
                const int32_t *nt = p.dev.notice + static_cast<int64_t>(k) * 2 * R;
                bool bad = false;
                if (G == 1 || ctr_smem != nullptr) {
                    // single-row messages, or counters in shared memory
                    int2 lhs[kNoticeLoads];   // kNoticeLoads destinations' notices in flight at once
                    for (int i = 0; i < nd; ++i) {
                        const int d = c + i * C;
                        if (i % kNoticeLoads == 0) {
#pragma unroll
                            for (int b = 0; b < kNoticeLoads; ++b)
                                lhs[b] = i + b < nd ? __ldcg(reinterpret_cast<const int2 *>(nt + 2 * (d + b * C)))
                                                    : make_int2(-1, -1);
                        }
                        int2 lh = lhs[0];
#pragma unroll
                        for (int b = 1; b < kNoticeLoads; ++b)
                            if (i % kNoticeLoads == b) lh = lhs[b];
                        int2 r = make_int2(0, 0);
                        MsgSpan sp;
                        if (lh.y >= 0 && !sp.init(lh, pt.cnt[s * R + d], pt.recv0[s * R + d], G)) {
                            bad = true;
                        } else if (lh.y >= 0) {
                            const int m0 = sp.sha || sp.shz ? msgoff[s * nd + i] : 0;
                            const unsigned olda = sp.sha ? add_half_counter(ctr_smem, m0 + sp.ga, sp.rowsa) : 0u;
                            const unsigned oldz = sp.shz ? add_half_counter(ctr_smem, m0 + sp.gz, sp.rowsz) : 0u;
                            bool fa, fz;
                            r = sp.posts(olda, oldz, fa, fz);
                        }
                        ranges[lane * ndmax + i] = r;
                        total += r.y - r.x;
                    }
                } else {
                    total = device_counter_spans(p.msg_rows, pt, R, C, G, c, s, nd, nt, ranges + lane * ndmax);
                    bad = total < 0;
                }
                if (bad) {
                    set_error(p.dev.err, EP_ERR_INVALID_ARG);
                    total = 0;
                }
            }
            __syncwarp();
            // Post the group's commands.  Each lane lists its own chunk's next
            // commands (at most kListPerLane) into the warp's list, packed the way
            // a slot holds them; the warp then posts the list, 32 (whole batches)
            // a round, one command per lane.  A batch may span chunks.
            int left = total;            // this lane's commands not yet listed
            int ci = 0, cm = 0;          // cursor: destination index, message past gb
            const int s_lane = take_now ? chunk_src(p, k) : 0;
            while (!failed) {
                const int take = min(left, kListPerLane);
                int incl = take;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                const int ltot = __shfl_sync(kFull, incl, 31);
                if (ltot == 0) break;
                for (int q = 0, at = incl - take; q < take; ++q, ++at) {
                    int2 g = ranges[lane * ndmax + ci];
                    while (cm >= g.y - g.x) {
                        ++ci;
                        cm = 0;
                        g = ranges[lane * ndmax + ci];
                    }
                    const int d = c + ci * C, pi = s_lane * R + d;
                    const int j0 = (g.x + cm) * G;
                    const int rows = min(G, pt.cnt[pi] - j0);
                    st_shared_v2(list + 2 * at,
                                 (static_cast<unsigned long long>(d) << 42) | (static_cast<unsigned long long>(rows) << 31) |
                                     static_cast<unsigned long long>(pt.send0[pi] + j0),
                                 static_cast<unsigned long long>(pt.recv0[pi] + j0));
                    ++cm;
                }
                left -= take;
                __syncwarp();
                for (int r0 = 0; r0 < ltot && !failed; r0 += rs) {
                    const int nround = min(rs, ltot - r0);
                    const bool mine = lane < nround;
                    unsigned long long w0 = 0ull, w1 = 0ull;
                    if (mine) {
                        const ulonglong2 v = ld_shared_v2(list + 2 * (r0 + lane));
                        w0 = v.x;
                        w1 = v.y;
                    }
                    // batch leaders reserve; every lane learns its batch's base
                    const int n = mine ? min(p.batch, nround - leader) : 0;
                    unsigned long long base = 0ull;
                    if (mine && lane == leader) base = atomicAdd(head, static_cast<unsigned long long>(n));
                    base = __shfl_sync(kFull, base, leader);
                    const unsigned long long idx = base + static_cast<unsigned long long>(lane - leader);
                    bool pending = mine;
                    uint64_t t0 = globaltimer_ns();
                    unsigned sleep = 32;
                    unsigned long long stalls = 0;
                    while (true) {
                        if (pending) {
                            const unsigned long long tail = ld_acquire_cta_shared(&words[kWProgress]);
                            if (base + n - tail <= limit) {
                                const unsigned long long lt = lap_tag(idx, p.lg_depth);
                                st_shared_v2(ring + 2 * (idx & dmask), w0 | lt, w1 | lt);
                                if (lane == leader) {
                                    st.batches += 1;
                                    st.max_batch = max(st.max_batch, static_cast<unsigned>(n));
                                    st.max_inflight = max(st.max_inflight, static_cast<unsigned>(base + n - tail));
                                    st.stalls += stalls;
                                }
                                pending = false;
                            } else {
                                ++stalls;
                            }
                        }
                        if (!__any_sync(kFull, pending)) break;
                        // waiting touches shared memory only; the device error word
                        // (an L2 round trip) is read every few tens of microseconds
                        bool give_up = false;
                        if (pending) {
                            const uint64_t now = globaltimer_ns();
                            if (now - t0 > p.timeout_ns) {
                                set_error(p.dev.err, EP_ERR_TIMEOUT);
                                give_up = true;
                            } else if (now - err_checked > kErrCheckNs) {
                                err_checked = now;
                                give_up = read_error(p.dev.err) != 0;
                            }
                        }
                        if (__any_sync(kFull, give_up)) {
                            failed = true;
                            break;
                        }
                        __nanosleep(sleep);
                        sleep = min(sleep * 2u, 64u);
                    }
                }
                __syncwarp();
            }
            // arrival signals: the pass's messages to each destination have
            // landed (their chunks' ready flags were acquired above) and are now
            // posted -- one fence per pass, then one add per destination
            if (!failed) {
                __syncwarp();
                if (lane == 0) fence_acq_rel_gpu();
                for (int i = 0; i < nd; ++i) {
                    int m = 0;
                    if (take_now) {
                        const int2 g = ranges[lane * ndmax + i];
                        m = g.y - g.x;
                    }
#pragma unroll
                    for (int o = 16; o; o >>= 1) m += __shfl_xor_sync(kFull, m, o);
                    if (lane == 0 && m > 0) red_add_relaxed(p.dev.signal + c + i * C, static_cast<unsigned long long>(m));
                }
            }
            __syncwarp();
        }
    }
    // statistics: one reduction per warp
    unsigned long long b = st.batches, sp = st.stalls;
    unsigned mb = st.max_batch, mi = st.max_inflight;
    for (int o = 16; o; o >>= 1) {
        b += __shfl_xor_sync(kFull, b, o);
        sp += __shfl_xor_sync(kFull, sp, o);
        mb = max(mb, __shfl_xor_sync(kFull, mb, o));
        mi = max(mi, __shfl_xor_sync(kFull, mi, o));
    }
    if (lane == 0 && b) {
        RingStatsDev *stt = p.dev.stats + c;
        atomicAdd(&stt->batches, b);
        atomicMax(&stt->max_batch, mb);
        atomicMax(&stt->max_inflight, mi);
        if (sp) atomicAdd(&stt->stall_polls, sp);
    }
}

// ------------------------------------------------------ channel CTA: poller
// Takes the longest run of published slots from the tail, copies the packed
// records into a shared staging ring for the logger, and moves the ring's
// tail (the retire point) in shared memory -- the posters read it there, so
// flow control costs no round trip.  Having no global stores of its own, its
// release on the tail waits on nothing slow.
__device__ void consumer_poll(const DispatchParams &p, long long expected, unsigned long long *words,
                              const unsigned long long *ring, unsigned long long *stage) {
    const int lane = threadIdx.x & 31;
    const unsigned long long base = words[kWBase];
    const unsigned long long end = base + static_cast<unsigned long long>(expected);
    int window = max(p.drain_batch, ((p.max_inflight + 31) / 32) * 32);
    window = min(window, 32 * kMaxPollRounds);
    const unsigned long long dmask = static_cast<unsigned long long>(p.D - 1);
    unsigned long long pos = base;
    uint64_t idle_since = globaltimer_ns(), err_checked = idle_since;
    unsigned sleep = 32;
    while (pos < end) {
        const int avail = static_cast<int>(min(end - pos, static_cast<unsigned long long>(window)));
        ulonglong2 v[kMaxPollRounds];
        bool pub[kMaxPollRounds];
#pragma unroll
        for (int q = 0; q < kMaxPollRounds; ++q) {
            pub[q] = false;
            v[q] = make_ulonglong2(0ull, 0ull);
            const int off = q * 32 + lane;
            if (off < avail) {
                const unsigned long long idx = pos + static_cast<unsigned long long>(off);
                v[q] = ld_shared_v2(ring + 2 * (idx & dmask));
                const unsigned long long lt = lap_tag(idx, p.lg_depth);
                pub[q] = (v[q].x & 0xFFFF000000000000ull) == lt && (v[q].y & 0xFFFF000000000000ull) == lt;
            }
        }
        int ready = 0;
#pragma unroll
        for (int q = 0; q < kMaxPollRounds; ++q) {
            if (ready < q * 32) break;
            const unsigned bal = __ballot_sync(kFull, pub[q]);
            ready += bal == kFull ? 32 : __ffs(~bal) - 1;
        }
        // room in the staging ring (the logger frees it as it writes the log)
        if (ready > 0 && pos + ready - ld_acquire_cta_shared(&words[kWLogged]) > kLogStage) ready = 0;
        if (ready > 0) {
#pragma unroll
            for (int q = 0; q < kMaxPollRounds; ++q) {
                const int off = q * 32 + lane;
                if (off < ready) {
                    const unsigned long long i = (pos - base + off) & (kLogStage - 1);
                    st_shared_v2(stage + 2 * i, v[q].x, v[q].y);
                }
            }
            pos += static_cast<unsigned long long>(ready);
            __syncwarp();
            if (lane == 0) st_release_cta_shared(&words[kWProgress], pos);   // slots read, records staged
            idle_since = globaltimer_ns();
            sleep = 32;
        } else {
            const uint64_t now = globaltimer_ns();
            if (now - idle_since > p.timeout_ns) {
                set_error(p.dev.err, EP_ERR_TIMEOUT);
                break;
            }
            if (now - err_checked > kErrCheckNs) {   // see the posters: an L2 round trip
                err_checked = now;
                if (read_error(p.dev.err) != 0) break;
            }
            __nanosleep(sleep);
            sleep = min(sleep * 2u, 128u);
        }
    }
    __syncwarp();
    if (lane == 0) st_release_cta_shared(&words[kWStopped], 1ull);
}

// ------------------------------------------------------ channel CTA: logger
// Decodes staged records into TransferCmds, appends them to the channel's log
// in device memory, and publishes the ring's cumulative tail (and, at the end,
// head) to device memory with release stores, for the host and the next call.
__device__ void consumer_log(const DispatchParams &p, int c, long long expected, unsigned long long *words,
                             const unsigned long long *stage) {
    const int lane = threadIdx.x & 31;
    unsigned long long *tail = p.dev.tail + static_cast<int64_t>(c) * kHeadStride;
    const unsigned long long base = words[kWBase];
    const unsigned long long end = base + static_cast<unsigned long long>(expected);
    const int64_t B = p.row_bytes;
    ep_transfer_cmd *log = p.dev.log + static_cast<int64_t>(c) * p.log_cap;
    unsigned long long logged = base;
    uint64_t idle_since = globaltimer_ns();
    while (logged < end) {
        const unsigned long long cur = ld_acquire_cta_shared(&words[kWProgress]);
        if (cur > logged) {
            for (unsigned long long j = logged + lane; j < cur; j += 32) {
                const unsigned long long i = (j - base) & (kLogStage - 1);
                const ulonglong2 w = ld_shared_v2(stage + 2 * i);
                const uint32_t d = static_cast<uint32_t>((w.x >> 42) & 63ull);
                const uint32_t rows = static_cast<uint32_t>((w.x >> 31) & 2047ull);
                const uint64_t src = (w.x & 0x7FFFFFFFull) * static_cast<uint64_t>(B);
                const uint64_t dst = (w.y & 0x7FFFFFFFull) * static_cast<uint64_t>(B);
                uint4 *o = reinterpret_cast<uint4 *>(log + (j - base));
                o[0] = make_uint4(d, rows * static_cast<uint32_t>(B), static_cast<uint32_t>(src),
                                  static_cast<uint32_t>(src >> 32));
                o[1] = make_uint4(static_cast<uint32_t>(dst), static_cast<uint32_t>(dst >> 32), 0u, 0u);
            }
            logged = cur;
            __syncwarp();
            if (lane == 0) {
                st_release_cta_shared(&words[kWLogged], logged);   // staging entries free again
                st_release(tail, logged);
            }
            idle_since = globaltimer_ns();
            continue;
        }
        if (ld_acquire_cta_shared(&words[kWStopped]) != 0ull &&
            ld_acquire_cta_shared(&words[kWProgress]) == logged)   // the poller stopped early
            break;
        if (globaltimer_ns() - idle_since > 2 * p.timeout_ns) {
            set_error(p.dev.err, EP_ERR_TIMEOUT);
            break;
        }
        __nanosleep(64);
    }
    __syncwarp();
    if (lane == 0) {
        p.dev.log_count[c] = static_cast<int64_t>(logged - base);
        // every command of the call has been reserved once all were retired
        st_release(p.dev.head + static_cast<int64_t>(c) * kHeadStride, atomicAdd(&words[kWHead], 0ull));
    }
}

__global__ void __launch_bounds__(kThreads, 1) dispatch_kernel(const DispatchParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const SmemLayout L(p.R, p.C, p.D, p.stage_bytes, p.stages, p.poster_warps, p.G);
    int *rbase = reinterpret_cast<int *>(smem + L.scratch_off);
    unsigned long long *words =
        reinterpret_cast<unsigned long long *>(smem + L.scratch_off + ((p.R + 3) & ~3) * 4);
    int *ids = reinterpret_cast<int *>(words + kNumWords);
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    Bars bars;
    bars.stage_full = b;
    bars.meta_full = b + p.stages;
    bars.meta_free = bars.meta_full + kMetaSlots;
    bars.stage_empty = bars.meta_free + kMetaSlots;
    int4 *item_info = reinterpret_cast<int4 *>(smem + L.info_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool channel_cta = static_cast<int>(blockIdx.x) < p.C;

    // Prologue: barriers, window starts, and the checks every CTA takes alike
    // so that either all of them run or none does.  Per-channel message
    // counts (for each ring's drain and the log capacity check) are summed by
    // every thread at once into shared counters: one round of loads, not a
    // dependent load per channel and destination.
    unsigned *chan = reinterpret_cast<unsigned *>(smem + L.chan_off);   // [C], prologue only
    long long n_recv = 0;
    int err0 = 0;
    if (threadIdx.x < p.C) chan[threadIdx.x] = 0u;
    // the first round of message-count loads, issued with the other prologue
    // loads (one round trip for all of them); summed after the barrier
    const int npairs = (p.s1 - p.s0) * p.R;
    const int32_t *mc = p.msg_count + static_cast<int64_t>(p.s0) * p.R;
    int v0[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = static_cast<int>(threadIdx.x) + q * kThreads;
        v0[q] = i < npairs ? __ldg(mc + i) : 0;
    }
    if (warp == 0 && lane == 0) {
        err0 = read_error(p.dev.err);
        if (!channel_cta) {
            const int store_warps = p.vec_store ? p.store_warps : 1;
            for (int i = 0; i < p.stages; ++i) {
                mbar_init(&bars.stage_full[i], 1);
                mbar_init(&bars.stage_empty[i], store_warps);
            }
            for (int i = 0; i < kMetaSlots; ++i) {
                mbar_init(&bars.meta_full[i], 1);
                mbar_init(&bars.meta_free[i], store_warps);
            }
            mbar_fence_init();
        }
        for (int i = 0; i < kNumWords; ++i) words[i] = 0ull;
        const int rb_last = __ldg(p.recv_base + p.R - 1), rc_last = __ldg(p.recv_count + p.R - 1);
        words[kWGen] = ld_relaxed_u32(p.dev.disp_gen);
        n_recv = static_cast<long long>(rb_last) + rc_last;
        if (channel_cta) {
            // the ring is drained between calls, so tail is where this call starts
            const unsigned long long base = ld_relaxed(p.dev.tail + static_cast<int64_t>(blockIdx.x) * kHeadStride);
            words[kWBase] = base;
            words[kWProgress] = base;
            words[kWHead] = base;
            words[kWLogged] = base;
        }
    }
    if (warp == 1)
        for (int d = lane; d < p.R; d += 32) rbase[d] = __ldg(p.recv_base + d);
    if (channel_cta) {
        // the ring: tags are laps of the cumulative index, so clear the slots
        // (a fresh launch's shared memory holds anything)
        unsigned long long *ring = reinterpret_cast<unsigned long long *>(smem + SmemLayout::ring_off(p.R));
        for (int i = threadIdx.x; i < 2 * p.D; i += blockDim.x) ring[i] = 0ull;
        int *tab = reinterpret_cast<int *>(smem);
        const int RR = p.R * p.R;
        for (int i = threadIdx.x; i < RR; i += blockDim.x) {
            tab[i] = __ldg(p.cnt + i);
            tab[RR + i] = __ldg(p.recv_off + i);
            tab[2 * RR + i] = __ldg(p.send_off + i);
        }
    }
    __syncthreads();
    for (int i0 = threadIdx.x; i0 < npairs; i0 += 4 * kThreads) {
        int v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            v[q] = i0 == static_cast<int>(threadIdx.x) ? v0[q]
                   : (i0 + q * kThreads < npairs ? __ldg(mc + i0 + q * kThreads) : 0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (v[q] != 0) atomicAdd(&chan[((i0 + q * kThreads) % p.R) % p.C], static_cast<unsigned>(v[q]));
    }
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // N against the receive capacity; every channel's count against its log
        long long worst = 0;
        for (int c = 0; c < p.C; ++c) worst = max(worst, static_cast<long long>(chan[c]));
        int abort = err0 != 0;
        if (n_recv > p.cap_rows || n_recv < 0) {
            set_error(p.dev.err, EP_ERR_CAPACITY);
            abort = 1;
        }
        if (worst > p.log_cap) {
            set_error(p.dev.err, EP_ERR_INVALID_ARG);
            abort = 1;
        }
        words[kWAbort] = static_cast<unsigned long long>(abort);
        words[kWExpected] = channel_cta ? static_cast<unsigned long long>(chan[blockIdx.x]) : 0ull;
    }
    __syncthreads();
    if (channel_cta && p.G > 1) {
        // message counters of this ring: the first one of each
        // pair (s, d), d = c + i*C, in (s, i) order, then one 16-bit counter
        // per message, in shared memory if they fit; else the device-memory
        // counters are used
        const int c = blockIdx.x;
        const int nd = c < p.R ? (p.R - 1 - c) / p.C + 1 : 0;
        const int coff = SmemLayout::counters_off(p.R, p.C, p.D, p.poster_warps);
        // counters are 16-bit halves of a word
        const long long room = 2 * (static_cast<long long>(L.scratch_off - coff) / 4 - static_cast<long long>(p.R) * nd);
        if (warp == 1) {
            int *msgoff = reinterpret_cast<int *>(smem + coff);
            const int *cntt = reinterpret_cast<const int *>(smem);
            int run = 0;
            for (int b0 = 0; room >= 0 && b0 < p.R * nd; b0 += 32) {
                const int idx = b0 + lane;
                int m = 0;
                if (idx < p.R * nd) {
                    const int sr = idx / nd, i = idx - sr * nd;
                    m = (cntt[sr * p.R + c + i * p.C] + p.G - 1) / p.G;
                }
                int incl = m;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                if (idx < p.R * nd) msgoff[idx] = run + incl - m;
                run += __shfl_sync(kFull, incl, 31);
            }
            if (lane == 0)
                words[kWCounters] = !(p.debug & EP_DEBUG_DEVICE_COUNTERS) && room >= 0 && run <= room
                                        ? static_cast<unsigned long long>(run) + 1ull
                                        : 0ull;
        }
        __syncthreads();
        if (words[kWCounters] != 0ull) {
            unsigned *ctr = reinterpret_cast<unsigned *>(smem + coff) + p.R * nd;
            const int n = static_cast<int>((words[kWCounters] - 1ull + 1ull) / 2);   // words of two counters
            for (int i = threadIdx.x; i < n; i += blockDim.x) ctr[i] = 0u;
            __syncthreads();
        }
    }
    const long long expected = static_cast<long long>(words[kWExpected]);

    if (words[kWAbort] == 0ull) {
        if (channel_cta) {
            const int c = blockIdx.x;
            if (warp != kPollWarp && warp != kLogWarp) {
                PairTables pt;
                pt.cnt = reinterpret_cast<const int *>(smem);
                pt.recv0 = pt.cnt + p.R * p.R;
                pt.send0 = pt.recv0 + p.R * p.R;
                const int pw = poster_index(warp);
                uint8_t *rb = smem + SmemLayout::ranges_off(p.R, p.D) + pw * SmemLayout::ranges_bytes_per_warp(p.R, p.C);
                uint8_t *lb =
                    smem + SmemLayout::lists_off(p.R, p.C, p.D, p.poster_warps) + pw * SmemLayout::kListBytesPerWarp;
                if (pw < p.poster_warps)
                poster_warp(p, c, pw, words, pt, reinterpret_cast<unsigned long long *>(smem + SmemLayout::ring_off(p.R)),
                            reinterpret_cast<int2 *>(rb), reinterpret_cast<unsigned long long *>(lb),
                            reinterpret_cast<int *>(smem + SmemLayout::counters_off(p.R, p.C, p.D, p.poster_warps)));
            } else if (!(p.debug & EP_DEBUG_DISABLE_CONSUMER)) {
                unsigned long long *ring = reinterpret_cast<unsigned long long *>(smem + SmemLayout::ring_off(p.R));
                unsigned long long *stage = ring + 2 * p.D;
                if (warp == kPollWarp)
                    consumer_poll(p, expected, words, ring, stage);
                else
                    consumer_log(p, c, expected, words, stage);
            }
        } else {
            if (warp == 0 && p.vec_store)
                copy_warp_vec(p, smem, L, bars, words, ids, item_info);
            else if (warp == 0)
                copy_warp(p, smem, L, bars, words, ids);
            else if (warp >= kStoreWarp0 && p.vec_store)
                store_warp(p, smem, L, bars, words, item_info, warp - kStoreWarp0);
            else if (warp == 1)
                meta_warp(p, smem, L, bars, rbase, words, ids);
            else if (warp == 2)
                notify_warp(p, words, ids);
        }
    }

    // Epilogue: the last CTA out advances the dispatch generation (which tags
    // the chunks' ready flags) and re-arms the counters for the next call.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.dev.disp_done, 1u) == gridDim.x - 1) {
            *p.dev.disp_done = 0u;
            *p.dev.chunk_next = 0u;
            atomicAdd(p.dev.disp_gen, 1u);
        }
    }
}

}  // namespace

// Geometry: one CTA per SM (C channel CTAs, the rest copy CTAs); stages sized
// so that a stage holds a run of whole rows (rows <= 16 KB) or one piece of a
// row, and as many stages as fit.
ep_status plan_dispatch(ep_ctx *h) {
    const int R = h->cfg.num_ranks, C = h->cfg.channels;
    const int64_t B = 2ll * h->cfg.hidden;
    const int kTargetStage = 16384;
    // Chunk size: about four chunks per copy CTA, so that the dynamic draw
    // balances the load even when the batch is small, 4 to 32 tokens (the
    // meta warp takes one token per lane).
    const int64_t T = static_cast<int64_t>(R) * h->cfg.tokens_per_rank;
    h->disp_grid = h->cfg.num_sms > 0 && h->cfg.num_sms < h->sm_count ? h->cfg.num_sms : h->sm_count;
    if (h->disp_grid < C + 1) return EP_ERR_INVALID_ARG;   // at least one copy CTA
    const int64_t copy_ctas = h->disp_grid - C;
    int chunk_tokens = kChunkTokens;
    while (chunk_tokens > 4 && T < 4 * copy_ctas * chunk_tokens) chunk_tokens /= 2;
    int rows_per_item = 1, pieces = 1, piece_bytes = static_cast<int>(B);
    if (B <= kTargetStage) {
        rows_per_item = static_cast<int>(kTargetStage / B);
        if (rows_per_item > chunk_tokens) rows_per_item = chunk_tokens;
        piece_bytes = static_cast<int>(B);
    } else {
        pieces = static_cast<int>((B + kTargetStage - 1) / kTargetStage);
        piece_bytes = static_cast<int>(((B + pieces - 1) / pieces + 15) / 16 * 16);
    }
    const int stage_bytes = ((rows_per_item * piece_bytes) + 127) / 128 * 128;
    int max_smem = 0;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess)
        return EP_ERR_CUDA;
    const int reserve = 1024;   // static + alignment slack
    // the most poster warps that fit, then the most stages
    int stages = 0, npw = kPosterWarpsMax;
    for (; npw >= 1 && stages == 0; npw /= 2) {
        for (int s = kStagesMax; s >= 3; --s) {
            SmemLayout L(R, C, h->cfg.ring_depth, stage_bytes, s, npw, static_cast<int>(h->G));
            if (L.total + reserve <= max_smem) {
                stages = s;
                break;
            }
        }
        if (stages) break;
    }
    if (stages == 0) return EP_ERR_INVALID_ARG;
    SmemLayout L(R, C, h->cfg.ring_depth, stage_bytes, stages, npw, static_cast<int>(h->G));
    h->poster_warps = npw;
    h->rows_per_item = rows_per_item;
    h->vec_store = (pieces == 1 && B <= kVecRowMax) ? 1 : 0;
    h->pieces = pieces;
    h->piece_bytes = piece_bytes;
    h->stage_bytes = stage_bytes;
    h->stages = stages;
    h->prefetch = kPrefetchItems < stages - 1 ? kPrefetchItems : stages - 1;
    h->store_lag = kStoreLagItems < stages - h->prefetch ? kStoreLagItems : stages - h->prefetch;
    h->meta_slots = kMetaSlots;
    h->disp_smem = static_cast<size_t>(L.total);
    h->disp_threads = kThreads;
    h->chunk_tokens = chunk_tokens;
    // With big chunks of 16 tokens or more on the TMA path, the last tokens of
    // every rank go in small chunks (a quarter of the big size), about
    // kSmallPerCta of them per copy CTA over the layer: they are drawn last,
    // so the copy CTAs finish within a small chunk of each other.  (Measured
    // slower elsewhere: 1-token chunks, and 8-token chunks of small rows.)
    const int Tpr = h->cfg.tokens_per_rank;
    const bool tiers = chunk_tokens >= 16 && B > kVecRowMax;
    const int small_tokens = tiers ? chunk_tokens / 4 : chunk_tokens;
    const int64_t tail_target = tiers ? (static_cast<int64_t>(kSmallPerCta) * copy_ctas * small_tokens + R - 1) / R : 0;
    const int big_tok = Tpr > tail_target ? static_cast<int>((Tpr - tail_target) / chunk_tokens) * chunk_tokens : 0;
    h->small_tokens = small_tokens;
    h->nbig = big_tok / chunk_tokens;
    h->nsmall = (Tpr - big_tok + small_tokens - 1) / small_tokens;
    h->nchunks = (h->nbig + h->nsmall) * R;
    if (cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(h->disp_smem)) != cudaSuccess)
        return EP_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel, kThreads, h->disp_smem) !=
            cudaSuccess ||
        per_sm < 1)
        return EP_ERR_CUDA;
    return EP_OK;
}

ep_status launch_dispatch(ep_ctx *h, const void *x, const ep_layout_out *lay, void *recv, int64_t cap_rows,
                          int s_begin, int s_end, cudaStream_t st) {
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
    p.msg_rows = h->dev.msg_rows;
    p.nbig = h->nbig;
    p.nsmall = h->nsmall;
    p.small_tokens = h->small_tokens;
    p.chunk_tokens = h->chunk_tokens;
    p.nchunks = h->nchunks;
    p.s0 = s_begin;
    p.s1 = s_end;
    p.nk = (s_end - s_begin) * (h->nbig + h->nsmall);
    p.rows_per_item = h->rows_per_item;
    p.pieces = h->pieces;
    p.piece_bytes = h->piece_bytes;
    p.stage_bytes = h->stage_bytes;
    p.stages = h->stages;
    p.prefetch = h->prefetch;
    p.store_lag = h->store_lag;
    p.meta_slots = h->meta_slots;
    p.slot_vec = (p.R % 4 == 0 && reinterpret_cast<uintptr_t>(lay->token_slot) % 16 == 0) ? 1 : 0;
    p.lg_depth = __builtin_ctz(static_cast<unsigned>(p.D));
    p.vec_store = h->vec_store;
    p.poster_warps = h->poster_warps;
    p.store_warps = kThreads / 32 - kStoreWarp0;
    void *args[] = {&p};
    const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(dispatch_kernel),
                                                      dim3(h->disp_grid), dim3(kThreads), args, h->disp_smem, st);
    return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace ep
