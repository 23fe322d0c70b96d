// ep_api.cu -- host side of the libep C ABI (declared in include/ep.h):
// configuration checks, the one device allocation a handle owns, launches,
// status and statistics.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "ep_internal.cuh"

using ep::DevState;

namespace ep {

// True if the kernels may dereference p on `device`: memory of that device,
// managed memory, or page-locked host memory mapped into the device's address
// space.  Pageable host memory, memory of another device and addresses the
// runtime does not know are refused, so that a wrong pointer is an
// EP_ERR_INVALID_ARG on the host instead of a fault on the GPU.
bool ptr_usable_on(int device, const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();   // not sticky; leave no error behind
        return false;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice: return a.device == device && a.devicePointer != nullptr;
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return a.devicePointer != nullptr;
    default: return false;
    }
}

// Rows per message: 8 when a bf16 row is under the 7 KB packing threshold
// (UCCL-EP article s4.1; batch size 8 from s5.3), else 1.
int default_rows_per_msg(int hidden) { return 2 * hidden < 7 * 1024 ? 8 : 1; }

}  // namespace ep

using ep::default_rows_per_msg;

namespace {

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ep_status cuda_ok(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

// Makes the handle's device current for one call and then puts the caller's
// back, so that a call made while another device is current still launches
// where the handle's memory lives.
struct DeviceGuard {
    int prev = -1;
    bool switched = false, ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev) {
            ok = cudaSetDevice(dev) == cudaSuccess;
            switched = ok;
        }
    }
    ~DeviceGuard() {
        if (switched) (void)cudaSetDevice(prev);
    }
    DeviceGuard(const DeviceGuard &) = delete;
    DeviceGuard &operator=(const DeviceGuard &) = delete;
};

constexpr uint64_t kMaxWaitNs = 10000000000ull;   // longest ep_wait_signal: 10 s

bool layout_ptrs_ok(const ep_layout_out *o) {
    return o && o->num_tokens_per_expert && o->num_tokens_per_rank && o->is_token_in_rank && o->token_slot &&
           o->recv_off && o->send_off && o->msg_count && o->recv_count && o->recv_base && o->expert_off;
}

// The same check through a small per-thread cache keyed by device and
// pointer value: callers pass the same buffers call after call, so the
// runtime is asked once per buffer.
bool ptr_usable(ep_ctx *h, const void *p) {
    constexpr int kSlots = 64;
    struct Slot {
        uintptr_t ptr;
        int device;
    };
    thread_local Slot cache[kSlots] = {};
    const uintptr_t v = reinterpret_cast<uintptr_t>(p);
    Slot &slot = cache[((v >> 8) ^ (v >> 20)) % kSlots];
    if (slot.ptr == v && slot.device == h->device) return true;
    if (!ep::ptr_usable_on(h->device, p)) return false;
    slot = Slot{v, h->device};
    return true;
}

bool layout_ptrs_usable(ep_ctx *h, const ep_layout_out *o) {
    return ptr_usable(h, o->num_tokens_per_expert) && ptr_usable(h, o->num_tokens_per_rank) &&
           ptr_usable(h, o->is_token_in_rank) && ptr_usable(h, o->token_slot) && ptr_usable(h, o->recv_off) &&
           ptr_usable(h, o->send_off) && ptr_usable(h, o->msg_count) && ptr_usable(h, o->recv_count) &&
           ptr_usable(h, o->recv_base) && ptr_usable(h, o->expert_off);
}

// Carves one allocation into 256-byte aligned pieces.
struct Carver {
    size_t off = 0;
    template <typename T>
    size_t take(size_t count) {
        const size_t at = (off + 255) & ~size_t(255);
        off = at + count * sizeof(T);
        return at;
    }
};

}  // namespace

extern "C" {

ep_status ep_config_init(ep_config *cfg, int32_t num_ranks, int32_t tokens_per_rank, int32_t hidden,
                         int32_t num_experts, int32_t topk) {
    if (!cfg) return EP_ERR_INVALID_ARG;
    memset(cfg, 0, sizeof(*cfg));
    cfg->num_ranks = num_ranks;
    cfg->tokens_per_rank = tokens_per_rank;
    cfg->hidden = hidden;
    cfg->num_experts = num_experts;
    cfg->topk = topk;
    cfg->channels = 8;        // HT_CHANNELS
    cfg->ring_depth = 1024;   // FIFO_DEPTH
    cfg->max_inflight = 256;  // MAX_INFLIGHT
    cfg->batch = 8;           // up to 8 commands per batch
    cfg->rows_per_msg = 0;    // default rule
    cfg->drain_batch = 32;    // DRAIN_BATCH_SIZE
    cfg->debug_flags = 0;
    cfg->timeout_ns = ep::kDefaultTimeoutNs;
    return EP_OK;
}

ep_status ep_config_check(const ep_config *c) {
    if (!c) return EP_ERR_INVALID_ARG;
    if (c->num_ranks < 1 || c->num_ranks > ep::kMaxRanks) return EP_ERR_INVALID_ARG;
    if (c->tokens_per_rank < 1) return EP_ERR_INVALID_ARG;
    if (c->hidden < 8 || c->hidden % 8 != 0) return EP_ERR_INVALID_ARG;
    if (c->num_experts < c->num_ranks || c->num_experts % c->num_ranks != 0 || c->num_experts > 4096)
        return EP_ERR_INVALID_ARG;
    if (c->topk < 1 || c->topk > ep::kMaxTopk || c->topk > c->num_experts) return EP_ERR_INVALID_ARG;
    if (c->channels < 1 || c->channels > ep::kMaxChannels) return EP_ERR_INVALID_ARG;
    // rings live in shared memory: 16 bytes a slot
    if (!is_pow2(c->ring_depth) || c->ring_depth < 8 || c->ring_depth > 8192) return EP_ERR_INVALID_ARG;
    if (c->max_inflight < 8 || c->max_inflight > c->ring_depth) return EP_ERR_INVALID_ARG;
    if (c->batch < 1 || c->batch > 8) return EP_ERR_INVALID_ARG;
    if (c->rows_per_msg < 0 || c->rows_per_msg > 2047) return EP_ERR_INVALID_ARG;   // 11 bits in a ring slot
    if (c->drain_batch < 32 || c->drain_batch > 512 || c->drain_batch % 32 != 0) return EP_ERR_INVALID_ARG;
    if (c->debug_flags & ~(EP_DEBUG_DISABLE_CONSUMER | EP_DEBUG_DEVICE_COUNTERS)) return EP_ERR_INVALID_ARG;
    if (c->num_sms < 0 || (c->num_sms > 0 && c->num_sms < c->channels + 1) || c->reserved != 0)
        return EP_ERR_INVALID_ARG;
    const int64_t T = static_cast<int64_t>(c->num_ranks) * c->tokens_per_rank;
    const int64_t kmin = c->topk < c->num_ranks ? c->topk : c->num_ranks;
    // receive rows are counted in int32
    if (T * kmin >= (1ll << 31) || T * c->num_ranks >= (1ll << 40)) return EP_ERR_INVALID_ARG;
    const int G = c->rows_per_msg ? c->rows_per_msg : default_rows_per_msg(c->hidden);
    // a message's byte size is a uint32
    if (static_cast<int64_t>(G) * 2 * c->hidden >= (1ll << 32)) return EP_ERR_INVALID_ARG;
    return EP_OK;
}

const char *ep_status_str(ep_status s) {
    switch (s) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
        case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
        case EP_ERR_CUDA: return "EP_ERR_CUDA";
        case EP_ERR_NOT_READY: return "EP_ERR_NOT_READY";
    }
    return "EP_ERR_UNKNOWN";
}

ep_status ep_create(const ep_config *cfg, ep_handle *out) {
    if (!out) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    ep_status st = ep_config_check(cfg);
    if (st != EP_OK) return st;
    ep_ctx *h = new (std::nothrow) ep_ctx();
    if (!h) return EP_ERR_INVALID_ARG;
    h->cfg = *cfg;
    if (h->cfg.timeout_ns == 0) h->cfg.timeout_ns = ep::kDefaultTimeoutNs;
    h->G = cfg->rows_per_msg ? cfg->rows_per_msg : default_rows_per_msg(cfg->hidden);
    const int R = cfg->num_ranks, E = cfg->num_experts, C = cfg->channels;
    const int64_t Tpr = cfg->tokens_per_rank, T = R * Tpr;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        delete h;
        return EP_ERR_CUDA;
    }
    h->tiles = static_cast<int>((T + ep::layout_tile(T) - 1) / ep::layout_tile(T));
    // log capacity: every message of every (s, d) with d in the busiest channel
    const int64_t ranks_per_chan = (R + C - 1) / C;
    const int64_t kmin = cfg->topk < ranks_per_chan ? cfg->topk : ranks_per_chan;
    h->log_cap = (T * kmin + h->G - 1) / h->G + static_cast<int64_t>(R) * ranks_per_chan;
    if ((st = ep::plan_dispatch(h)) != EP_OK || (st = ep::plan_combine(h)) != EP_OK ||
        (st = ep::plan_expert_layout(h)) != EP_OK) {
        delete h;
        return st;
    }

    Carver cv;
    const size_t o_err = cv.take<int32_t>(1);
    const size_t o_ticket = cv.take<unsigned long long>(1);
    const size_t o_done = cv.take<unsigned int>(1);
    const size_t o_desc = cv.take<unsigned long long>(static_cast<size_t>(h->tiles) * R);
    const size_t o_hist = cv.take<int32_t>(static_cast<size_t>(R) * E);
    const size_t o_pref = cv.take<int32_t>(static_cast<size_t>(R + 1) * R);
    const size_t o_nrecv = cv.take<int64_t>(1);
    const size_t o_head = cv.take<unsigned long long>(static_cast<size_t>(C) * ep::kHeadStride);
    const size_t o_tail = cv.take<unsigned long long>(static_cast<size_t>(C) * ep::kHeadStride);
    const size_t o_stats = cv.take<ep::RingStatsDev>(C);
    const size_t o_log = cv.take<ep_transfer_cmd>(static_cast<size_t>(C) * h->log_cap);
    const size_t o_lcount = cv.take<int64_t>(C);
    const size_t o_notice = cv.take<int32_t>(static_cast<size_t>(h->nchunks) * 2 * R);
    const size_t o_ready = cv.take<unsigned int>(static_cast<size_t>(h->nchunks));
    const size_t o_gen = cv.take<unsigned int>(1);
    const size_t o_ddone = cv.take<unsigned int>(1);
    const size_t o_cnext = cv.take<unsigned int>(1);
    const size_t o_signal = cv.take<unsigned long long>(R);
    const size_t o_xticket = cv.take<unsigned long long>(1);
    const size_t o_xdesc = cv.take<unsigned long long>(static_cast<size_t>(h->xtiles) * E);
    // rows landed per multi-row message that spans chunks, indexed by its first
    // send row (N <= T * min(K, R)); only messages of G > 1 rows span chunks
    const int64_t kmin_all = cfg->topk < R ? cfg->topk : R;
    const size_t o_msgrows = cv.take<unsigned int>(h->G > 1 ? static_cast<size_t>(T * kmin_all) : 0);
    h->alloc_bytes = cv.off;
    if (cudaMalloc(&h->alloc_base, h->alloc_bytes) != cudaSuccess) {
        delete h;
        return EP_ERR_CUDA;
    }
    if (cudaMemset(h->alloc_base, 0, h->alloc_bytes) != cudaSuccess) {
        cudaFree(h->alloc_base);
        delete h;
        return EP_ERR_CUDA;
    }
    uint8_t *b = static_cast<uint8_t *>(h->alloc_base);
    DevState &d = h->dev;
    d.err = reinterpret_cast<int32_t *>(b + o_err);
    d.ticket = reinterpret_cast<unsigned long long *>(b + o_ticket);
    d.done = reinterpret_cast<unsigned int *>(b + o_done);
    d.tile_desc = reinterpret_cast<unsigned long long *>(b + o_desc);
    d.hist = reinterpret_cast<int32_t *>(b + o_hist);
    d.col_prefix = reinterpret_cast<int32_t *>(b + o_pref);
    d.n_recv = reinterpret_cast<int64_t *>(b + o_nrecv);
    d.head = reinterpret_cast<unsigned long long *>(b + o_head);
    d.tail = reinterpret_cast<unsigned long long *>(b + o_tail);
    d.stats = reinterpret_cast<ep::RingStatsDev *>(b + o_stats);
    d.log = reinterpret_cast<ep_transfer_cmd *>(b + o_log);
    d.log_count = reinterpret_cast<int64_t *>(b + o_lcount);
    d.notice = reinterpret_cast<int32_t *>(b + o_notice);
    d.ready = reinterpret_cast<unsigned int *>(b + o_ready);
    d.disp_gen = reinterpret_cast<unsigned int *>(b + o_gen);
    d.disp_done = reinterpret_cast<unsigned int *>(b + o_ddone);
    d.chunk_next = reinterpret_cast<unsigned int *>(b + o_cnext);
    d.signal = reinterpret_cast<unsigned long long *>(b + o_signal);
    d.xticket = reinterpret_cast<unsigned long long *>(b + o_xticket);
    d.xdesc = reinterpret_cast<unsigned long long *>(b + o_xdesc);
    d.msg_rows = reinterpret_cast<unsigned int *>(b + o_msgrows);
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(h->alloc_base);
        delete h;
        return EP_ERR_CUDA;
    }
    *out = h;
    return EP_OK;
}

ep_status ep_destroy(ep_handle h) {
    if (!h) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    const cudaError_t e1 = cudaDeviceSynchronize();
    const cudaError_t e2 = cudaFree(h->alloc_base);
    delete h;
    return (e1 == cudaSuccess && e2 == cudaSuccess) ? EP_OK : EP_ERR_CUDA;
}

ep_status ep_last_device_status(ep_handle h, int32_t *code) {
    if (!h || !code) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return EP_ERR_CUDA;
    return cuda_ok(cudaMemcpy(code, h->dev.err, sizeof(int32_t), cudaMemcpyDeviceToHost));
}

ep_status ep_reset(ep_handle h) {
    if (!h) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return EP_ERR_CUDA;
    if (cudaMemset(h->alloc_base, 0, h->alloc_bytes) != cudaSuccess) return EP_ERR_CUDA;
    return cuda_ok(cudaDeviceSynchronize());
}

ep_status ep_layout(ep_handle h, const int32_t *topk_idx, const ep_layout_out *out, int64_t *n_recv_host,
                    void *stream) {
    if (!h || !topk_idx || !layout_ptrs_ok(out)) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (!ptr_usable(h, topk_idx) || !layout_ptrs_usable(h, out)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ep_status s = ep::launch_layout(h, topk_idx, out, st);
    if (s != EP_OK || !n_recv_host) return s;
    int64_t n = 0;
    if (cudaMemcpyAsync(&n, h->dev.n_recv, sizeof(n), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return EP_ERR_CUDA;
    *n_recv_host = n;
    return EP_OK;
}

ep_status ep_dispatch_ranks(ep_handle h, const void *x, const ep_layout_out *layout, void *recv,
                            int64_t recv_capacity_rows, int32_t src_begin, int32_t src_end, void *stream) {
    if (!h || !x || !recv || !layout_ptrs_ok(layout) || recv_capacity_rows < 0) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (src_begin < 0 || src_end < src_begin || src_end > h->cfg.num_ranks) return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv)) return EP_ERR_INVALID_ARG;
    if (!ptr_usable(h, x) || !ptr_usable(h, recv) || !layout_ptrs_usable(h, layout)) return EP_ERR_INVALID_ARG;
    return ep::launch_dispatch(h, x, layout, recv, recv_capacity_rows, src_begin, src_end,
                               static_cast<cudaStream_t>(stream));
}

ep_status ep_dispatch(ep_handle h, const void *x, const ep_layout_out *layout, void *recv,
                      int64_t recv_capacity_rows, void *stream) {
    return ep_dispatch_ranks(h, x, layout, recv, recv_capacity_rows, 0, h ? h->cfg.num_ranks : 0, stream);
}

ep_status ep_combine_tokens(ep_handle h, const void *expert_out, int64_t expert_out_rows, const float *topk_weights,
                            const int32_t *topk_idx, const ep_layout_out *layout, void *out, int64_t t_begin,
                            int64_t t_end, void *stream) {
    if (!h || !expert_out || !topk_weights || !topk_idx || !layout_ptrs_ok(layout) || !out || expert_out_rows < 0)
        return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    const int64_t T = static_cast<int64_t>(h->cfg.num_ranks) * h->cfg.tokens_per_rank;
    if (t_begin < 0 || t_end < t_begin || t_end > T) return EP_ERR_INVALID_ARG;
    if (!aligned16(expert_out) || !aligned16(out)) return EP_ERR_INVALID_ARG;
    if (!ptr_usable(h, expert_out) || !ptr_usable(h, topk_weights) || !ptr_usable(h, topk_idx) ||
        !ptr_usable(h, out) || !layout_ptrs_usable(h, layout))
        return EP_ERR_INVALID_ARG;
    return ep::launch_combine(h, expert_out, expert_out_rows, topk_weights, topk_idx, layout, out, t_begin, t_end,
                              static_cast<cudaStream_t>(stream));
}

ep_status ep_combine(ep_handle h, const void *expert_out, int64_t expert_out_rows, const float *topk_weights,
                     const int32_t *topk_idx, const ep_layout_out *layout, void *out, void *stream) {
    const int64_t T = h ? static_cast<int64_t>(h->cfg.num_ranks) * h->cfg.tokens_per_rank : 0;
    return ep_combine_tokens(h, expert_out, expert_out_rows, topk_weights, topk_idx, layout, out, 0, T, stream);
}

ep_status ep_expert_layout(ep_handle h, const int32_t *topk_idx, const float *topk_weights,
                           const ep_layout_out *layout, const ep_expert_layout_out *out, int64_t recv_rows,
                           int64_t expert_rows_capacity, void *stream) {
    if (!h || !topk_idx || !topk_weights || !layout_ptrs_ok(layout) || !out || !out->recv_topk_idx ||
        !out->recv_topk_weights || !out->recv_src_token || !out->expert_rows || !out->expert_count ||
        recv_rows < 0 || expert_rows_capacity < 0)
        return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (!ptr_usable(h, topk_idx) || !ptr_usable(h, topk_weights) || !layout_ptrs_usable(h, layout) ||
        !ptr_usable(h, out->recv_topk_idx) || !ptr_usable(h, out->recv_topk_weights) ||
        !ptr_usable(h, out->recv_src_token) || !ptr_usable(h, out->expert_rows) || !ptr_usable(h, out->expert_count))
        return EP_ERR_INVALID_ARG;
    return ep::launch_expert_layout(h, topk_idx, topk_weights, layout, out, recv_rows, expert_rows_capacity,
                                    static_cast<cudaStream_t>(stream));
}

ep_status ep_signal_ptr(ep_handle h, const uint64_t **signals) {
    if (!h || !signals) return EP_ERR_INVALID_ARG;
    *signals = reinterpret_cast<const uint64_t *>(h->dev.signal);
    return EP_OK;
}

ep_status ep_signal_get(ep_handle h, uint64_t *host_out, int32_t n) {
    if (!h || !host_out || n < 0 || n > h->cfg.num_ranks) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (n == 0) return EP_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) return EP_ERR_CUDA;
    return cuda_ok(cudaMemcpy(host_out, h->dev.signal, sizeof(uint64_t) * n, cudaMemcpyDeviceToHost));
}

ep_status ep_signal_reset(ep_handle h, void *stream) {
    if (!h) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    return cuda_ok(cudaMemsetAsync(h->dev.signal, 0, sizeof(uint64_t) * h->cfg.num_ranks,
                                   static_cast<cudaStream_t>(stream)));
}

ep_status ep_wait_signal(ep_handle h, int32_t dst_rank, uint64_t expected, uint64_t timeout_ns, int32_t *status_out,
                         void *stream) {
    if (!h || !status_out || dst_rank < 0 || dst_rank >= h->cfg.num_ranks || timeout_ns > kMaxWaitNs)
        return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (!ptr_usable(h, status_out)) return EP_ERR_INVALID_ARG;
    return ep::launch_wait_signal(h->dev.signal + dst_rank, expected, timeout_ns, status_out,
                                  static_cast<cudaStream_t>(stream));
}

ep_status ep_cmd_log_get(ep_handle h, ep_cmd_log *out) {
    if (!h || !out) return EP_ERR_INVALID_ARG;
    out->cmds = h->dev.log;
    out->count = h->dev.log_count;
    out->capacity_per_channel = h->log_cap;
    out->channels = h->cfg.channels;
    return EP_OK;
}

ep_status ep_ring_stats_get(ep_handle h, ep_ring_stats *out, int32_t n) {
    if (!h || !out || n < 0 || n > h->cfg.channels) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (n == 0) return EP_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) return EP_ERR_CUDA;
    const int C = h->cfg.channels;
    ep::RingStatsDev *st = static_cast<ep::RingStatsDev *>(malloc(sizeof(ep::RingStatsDev) * C));
    unsigned long long *hd = static_cast<unsigned long long *>(malloc(sizeof(unsigned long long) * C * ep::kHeadStride));
    unsigned long long *tl = static_cast<unsigned long long *>(malloc(sizeof(unsigned long long) * C * ep::kHeadStride));
    int64_t *lc = static_cast<int64_t *>(malloc(sizeof(int64_t) * C));
    ep_status rc = EP_OK;
    if (!st || !hd || !tl || !lc) rc = EP_ERR_INVALID_ARG;
    if (rc == EP_OK &&
        (cudaMemcpy(st, h->dev.stats, sizeof(ep::RingStatsDev) * C, cudaMemcpyDeviceToHost) != cudaSuccess ||
         cudaMemcpy(hd, h->dev.head, sizeof(unsigned long long) * C * ep::kHeadStride, cudaMemcpyDeviceToHost) !=
             cudaSuccess ||
         cudaMemcpy(tl, h->dev.tail, sizeof(unsigned long long) * C * ep::kHeadStride, cudaMemcpyDeviceToHost) !=
             cudaSuccess ||
         cudaMemcpy(lc, h->dev.log_count, sizeof(int64_t) * C, cudaMemcpyDeviceToHost) != cudaSuccess))
        rc = EP_ERR_CUDA;
    if (rc == EP_OK) {
        for (int c = 0; c < n; ++c) {
            out[c].head = hd[c * ep::kHeadStride];
            out[c].tail = tl[c * ep::kHeadStride];
            out[c].batches = st[c].batches;
            out[c].stall_polls = st[c].stall_polls;
            out[c].max_batch = st[c].max_batch;
            out[c].max_inflight = st[c].max_inflight;
            out[c].last_count = lc[c];
        }
    }
    free(st);
    free(hd);
    free(tl);
    free(lc);
    return rc;
}

ep_status ep_check_completion(ep_handle h, int32_t channel, uint64_t cmd_idx) {
    if (!h || channel < 0 || channel >= h->cfg.channels) return EP_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    if (!dg.ok) return EP_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return EP_ERR_CUDA;
    unsigned long long tail = 0;
    if (cudaMemcpy(&tail, h->dev.tail + static_cast<size_t>(channel) * ep::kHeadStride, sizeof(tail),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return EP_ERR_CUDA;
    // a command is complete once the consumer's tail has moved past it
    return tail > cmd_idx ? EP_OK : EP_ERR_NOT_READY;
}

ep_status ep_get_info(ep_handle h, ep_info *out) {
    if (!h || !out) return EP_ERR_INVALID_ARG;
    memset(out, 0, sizeof(*out));
    out->rows_per_msg = h->G;
    out->sm_count = h->sm_count;
    out->dispatch_grid = h->disp_grid;
    out->dispatch_stages = h->stages;
    out->dispatch_stage_bytes = h->stage_bytes;
    out->combine_grid = h->comb_grid;
    out->layout_tiles = h->tiles;
    out->dispatch_chunk_tokens = h->chunk_tokens;
    out->log_capacity_per_channel = h->log_cap;
    out->scratch_bytes = static_cast<int64_t>(h->alloc_bytes);
    return EP_OK;
}

}  // extern "C"
