// ep_internal.cuh -- shared pieces of the libep CUDA sources (sm_103a):
// the handle, the device state it owns, the launch parameter blocks, and
// thin inline-PTX wrappers (acquire/release accesses, %globaltimer, mbarrier,
// 1-D TMA bulk copies).  Host-visible API: include/ep.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep.h"

namespace ep {

// Limits the kernels are written for (also checked by ep_config_check).
constexpr int kMaxRanks = 64;
constexpr int kMaxTopk = 32;
constexpr int kMaxChannels = 64;
constexpr int kChunkTokens = 32;         // dispatch: most tokens per chunk (one per lane)
constexpr int kHeadStride = 16;          // u64s between two channels' head/tail words (128 B)
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// ---------------------------------------------------------------- device state

// Per-channel producer statistics (cumulative).  Matches the leading fields
// of ep_ring_stats; head/tail/last_count are stored elsewhere.
struct RingStatsDev {
    unsigned long long batches;
    unsigned long long stall_polls;
    unsigned int max_batch;
    unsigned int max_inflight;
};

// Device pointers the handle owns (one cudaMalloc, carved).
struct DevState {
    int32_t *err;                       // sticky error word (ep_status)
    // layout scan
    unsigned long long *ticket;         // tiles handed out so far (all calls)
    unsigned int *done;                 // tiles finished in the current call
    unsigned long long *tile_desc;      // [tiles * R] packed (epoch, flag, value)
    int32_t *hist;                      // [R * E] per-call histogram scratch, left zeroed
    int32_t *col_prefix;                // [(R + 1) * R] column prefix at each rank's first token
    int64_t *n_recv;                    // N of the last layout
    // rings
    unsigned long long *head;           // [C * kHeadStride]
    unsigned long long *tail;           // [C * kHeadStride]
    RingStatsDev *stats;                // [C]
    ep_transfer_cmd *log;               // [C * log_cap]
    int64_t *log_count;                 // [C]
    int32_t *notice;                    // [nchunks * 2R] per chunk: first/last window slot per rank
    unsigned int *ready;                // [nchunks] = dispatch generation + 1 once the chunk's rows landed
    unsigned int *disp_gen;             // dispatch calls so far (tags `ready`)
    unsigned int *disp_done;            // CTAs finished in the current dispatch
    unsigned int *chunk_next;           // next chunk to hand to a copy CTA in the current dispatch
    unsigned long long *signal;         // [R] messages landed per destination rank (cumulative)
    unsigned int *msg_rows;             // [T * min(K, R)] when G > 1: rows landed of a message that
                                        // spans chunks, at its first send row; zero between calls
    // expert layout scan
    unsigned long long *xticket;        // expert-layout tiles handed out so far (all calls)
    unsigned long long *xdesc;          // [xtiles * E] packed (epoch, flag, value)
};

// Layout kernel parameters.
struct LayoutParams {
    const int32_t *topk_idx;
    ep_layout_out out;
    DevState dev;
    int64_t T;
    int R, Tpr, E, K, Er, G;
    int tiles;
    int in_rank_vec;   // bytes per is_token_in_rank store: 16, 4 or 1
    int slot_vec;      // 1: token_slot rows take 16-byte stores
    int topk_vec4;     // 1: topk_idx rows take 16-byte loads
    int er_shift;      // log2(E / R) when it is a power of two, else -1
};

// Dispatch kernel parameters.
struct DispatchParams {
    const uint8_t *x;
    uint8_t *recv;
    int64_t cap_rows;
    const int32_t *token_slot, *recv_base, *recv_count, *recv_off, *send_off, *cnt, *msg_count;
    DevState dev;
    unsigned int *msg_rows;   // dev.msg_rows (G > 1)
    int64_t T;
    int64_t row_bytes;
    int64_t log_cap;
    uint64_t timeout_ns;
    int R, Tpr, C, D, max_inflight, batch, G, drain_batch, debug;
    // A source rank's tokens are cut into nbig chunks of chunk_tokens tokens,
    // then nsmall chunks of small_tokens (the last may be short).  Chunk ids:
    // big chunks rank-major [0, R*nbig), then small chunks rank-major; a call
    // draws its big chunks first, so the last work handed out is fine-grained.
    int nbig, nsmall, small_tokens, nchunks;
    int nk;              // chunks of this call: those of source ranks [s0, s1)
    int s0, s1;
    int chunk_tokens;    // tokens per big chunk (4..32)
    int rows_per_item;   // tokens per item when a row fits a stage, else 1
    int pieces;          // pieces per row when it does not, else 1
    int piece_bytes;     // bytes per piece (a multiple of 16)
    int stage_bytes;     // bytes per shared-memory stage
    int stages, prefetch, meta_slots;
    int store_lag;       // items whose bulk stores may be in flight
    int slot_vec;        // 1: token_slot rows are 16-byte aligned (int4 loads)
    int vec_store;       // 1: rows leave shared memory by the store warps' vector stores
    int store_warps;     // store warps per copy CTA on that path
    int poster_warps;    // poster warps per channel CTA that run (1..8)
    int lg_depth;        // log2(D)
};

// Combine kernel parameters.
struct CombineParams {
    const uint8_t *expert_out;
    int64_t eo_rows;
    const float *w;
    const int32_t *topk_idx, *token_slot, *recv_base;
    uint8_t *out;
    DevState dev;
    int64_t T;
    int64_t t_begin, t_end;   // tokens of this call
    int64_t row_bytes;
    int R, K, E, Er;
    int nseg;            // 16-byte segments per row
    int nparts;          // work items per token (parts of its row)
};

}  // namespace ep

// The opaque handle of the C ABI.
struct ep_ctx {
    ep_config cfg;
    int G;
    int device;
    int sm_count;
    ep::DevState dev;
    void *alloc_base;
    size_t alloc_bytes;
    int tiles;
    // dispatch geometry
    int disp_grid, disp_threads;
    size_t disp_smem;
    int stage_bytes, stages, prefetch, meta_slots, store_lag;
    int rows_per_item, pieces, piece_bytes;
    int nbig, nsmall, small_tokens, nchunks, chunk_tokens;
    int vec_store;
    int poster_warps;
    int64_t log_cap;
    // combine geometry
    int comb_grid, comb_threads;
    // expert layout geometry
    int xtiles;
};

namespace ep {

// Host launchers (one per kernel source file).
ep_status launch_layout(ep_ctx *h, const int32_t *topk_idx, const ep_layout_out *out,
                        cudaStream_t st);
ep_status launch_dispatch(ep_ctx *h, const void *x, const ep_layout_out *lay, void *recv,
                          int64_t cap_rows, int s_begin, int s_end, cudaStream_t st);
ep_status launch_combine(ep_ctx *h, const void *expert_out, int64_t eo_rows, const float *w,
                         const int32_t *topk_idx, const ep_layout_out *lay, void *out,
                         int64_t t_begin, int64_t t_end, cudaStream_t st);
ep_status launch_wait_signal(const unsigned long long *signal, unsigned long long expected,
                             unsigned long long timeout_ns, int32_t *status, cudaStream_t st);
ep_status launch_expert_layout(ep_ctx *h, const int32_t *topk_idx, const float *topk_weights,
                               const ep_layout_out *lay, const ep_expert_layout_out *out,
                               int64_t recv_rows, int64_t rows_cap, cudaStream_t st);
// Tokens per layout tile (one per thread) for T tokens (ep_layout.cu).
int layout_tile(int64_t T);
void fill_layout_vec(LayoutParams &p);
// Rows per message G when ep_config.rows_per_msg is 0 (ep_api.cu).
int default_rows_per_msg(int hidden);
// Dispatch geometry, decided once per handle.
ep_status plan_dispatch(ep_ctx *h);
ep_status plan_combine(ep_ctx *h);
ep_status plan_expert_layout(ep_ctx *h);

// ------------------------------------------------------------ device helpers
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32_(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void set_error(int32_t *err, int code) {
    atomicCAS(reinterpret_cast<int *>(err), 0, code);
}
__device__ __forceinline__ int read_error(const int32_t *err) {
    return *reinterpret_cast<const volatile int *>(err);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// atomic add with acquire and release semantics (GPU scope); returns the old value
__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// relaxed atomic add (GPU scope); returns the old value
__device__ __forceinline__ unsigned int atom_add_relaxed(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned int atom_add_acq_rel_cta_shared(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(v)
                 : "memory");
    return old;
}
__device__ __forceinline__ void red_add_relaxed(unsigned long long *p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(unsigned int *p, unsigned int v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_relaxed_v2(const unsigned long long *p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_v2(unsigned long long *p, unsigned long long a, unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_shared_v2(const unsigned long long *p) {
    ulonglong2 v;
    asm volatile("ld.volatile.shared::cta.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "r"(smem_u32_(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_v2(unsigned long long *p, unsigned long long a, unsigned long long b) {
    asm volatile("st.volatile.shared::cta.v2.u64 [%0], {%1, %2};" ::"r"(smem_u32_(p)), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_release_cta_shared(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.cta.shared::cta.u64 [%0], %1;" ::"r"(smem_u32_(p)), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_cta_shared(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.cta.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32_(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---- decoupled look-back (Merrill & Garland 2016), shared by the scans
// Descriptor word of one tile and column: {epoch:30 | flag:2 | value:32};
// flag 1 = the tile's aggregate, 2 = the inclusive prefix through the tile.
constexpr uint32_t kLookAggregate = 1u, kLookPrefix = 2u;
constexpr int kLookBatch = 8;   // predecessors read per round trip

__device__ __forceinline__ unsigned long long look_desc(uint32_t epoch, uint32_t flag, uint32_t value) {
    return (static_cast<unsigned long long>(epoch) << 34) | (static_cast<unsigned long long>(flag) << 32) | value;
}

// Exclusive prefix of `tile` in one column: walks back over the predecessors'
// descriptors (column entry c of tile t at desc[t * stride + c]), adding
// aggregates until an inclusive prefix is found.  kLookBatch descriptors are
// read per round trip; the walk stops at the first one not yet published in
// this epoch and polls it again.  Bounded by timeout_ns from t_start: on
// expiry it sets EP_ERR_TIMEOUT and returns what it has.
__device__ __forceinline__ int lookback_excl(const unsigned long long *desc, int64_t stride, int c, int tile,
                                             uint32_t epoch, uint64_t t_start, uint64_t timeout_ns, int32_t *err) {
    int excl = 0;
    int pred = tile - 1;
    uint32_t spins = 0;
    while (pred >= 0) {
        unsigned long long v[kLookBatch];
#pragma unroll
        for (int q = 0; q < kLookBatch; ++q)
            v[q] = pred - q >= 0 ? ld_relaxed(desc + static_cast<int64_t>(pred - q) * stride + c) : 0ull;
        bool found = false, stall = false;
#pragma unroll
        for (int q = 0; q < kLookBatch; ++q) {
            if (found || stall || pred < 0) continue;
            const uint32_t ep_v = static_cast<uint32_t>(v[q] >> 34);
            const uint32_t flag = static_cast<uint32_t>(v[q] >> 32) & 3u;
            if (ep_v == epoch && flag != 0u) {
                excl += static_cast<int>(static_cast<uint32_t>(v[q]));
                if (flag == kLookPrefix) found = true;
                --pred;
            } else {
                stall = true;
            }
        }
        if (found) break;
        if (stall && (++spins & 7u) == 0u) {
            if (globaltimer_ns() - t_start > timeout_ns) {
                set_error(err, EP_ERR_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
    }
    return excl;
}

// ---- mbarrier (shared::cta)
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Non-blocking test of phase `parity` (true once that phase has completed).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Potentially blocking (for a hardware-bounded time) wait on phase `parity`.
__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Reads a grid's error word at most once per kErrPollNs.  Waiting warps of
// every CTA poll it; read on every spin, that one word became the hottest
// line in L2 and slowed every access that shared its slice.
constexpr uint64_t kErrPollNs = 10000;
struct ErrPoll {
    uint64_t next;
    __device__ __forceinline__ explicit ErrPoll(uint64_t now) : next(now + kErrPollNs) {}
    __device__ __forceinline__ bool raised(const int32_t *err, uint64_t now) {
        if (now < next) return false;
        next = now + kErrPollNs;
        return read_error(err) != 0;
    }
};

// Bounded wait: true when the phase completed; false when the time limit ran
// out or (err != nullptr) another thread of the grid raised an error (seen
// within kErrPollNs).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, const int32_t *err,
                                                  uint64_t timeout_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    ErrPoll ep(t0);
    while (true) {
        if (mbar_try(bar, parity)) return true;
        const uint64_t now = globaltimer_ns();
        if (err != nullptr && ep.raised(err, now)) return false;
        if (now - t0 > timeout_ns) return false;
    }
}

// ---- 1-D TMA bulk copies (cp.async.bulk): 16-byte aligned addresses, sizes
// a multiple of 16.  Global -> shared completes on an mbarrier; shared ->
// global completes per bulk async-group of the issuing thread.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_s2g(void *gmem_dst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Runtime-N wait on this thread's bulk groups (N clamped to 0..15).
__device__ __forceinline__ void bulk_wait_n(int n) {
    switch (n) {
        case 0: bulk_wait<0>(); break;
        case 1: bulk_wait<1>(); break;
        case 2: bulk_wait<2>(); break;
        case 3: bulk_wait<3>(); break;
        case 4: bulk_wait<4>(); break;
        case 5: bulk_wait<5>(); break;
        case 6: bulk_wait<6>(); break;
        case 7: bulk_wait<7>(); break;
        case 8: bulk_wait<8>(); break;
        case 9: bulk_wait<9>(); break;
        case 10: bulk_wait<10>(); break;
        case 11: bulk_wait<11>(); break;
        case 12: bulk_wait<12>(); break;
        case 13: bulk_wait<13>(); break;
        case 14: bulk_wait<14>(); break;
        default: bulk_wait<15>(); break;
    }
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// generic-proxy accesses to shared memory before later async-proxy (TMA) ones
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared::cta.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32_(p))
                 : "memory");
    return v;
}

#endif  // __CUDACC__

}  // namespace ep
