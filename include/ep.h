/*
 * ep.h -- C ABI of libep: token layout, dispatch and combine of one MoE
 * expert-parallel (EP) layer on one GB300 GPU, with the EP group's R ranks
 * held as partitions of device buffers.
 *
 * Articles this interface follows:
 *  [UCCL-EP] "UCCL-EP: GPU-side FIFO queues and CPU proxy threads"
 *            (peacm.com/news/835744)
 *  [GIN]     "NCCL GIN: device-initiated GPU networking" (bjdmk.com.cn/news/2086017)
 *  [NOTES]   "GPU communication mechanisms and optimisation techniques"
 *            (blog.zhenwei.site)
 *
 * Conventions for every call:
 *  - All tensor arguments are DEVICE pointers owned by the caller (e.g. torch
 *    allocations); the library never frees them.  Row-major, dense.  Each
 *    call asks the CUDA runtime what every pointer is (cached per host thread
 *    by device and pointer value) and accepts memory of the handle's device,
 *    managed memory and page-locked host memory mapped into the device's
 *    address space; pageable host memory, another device's memory and unknown
 *    addresses are EP_ERR_INVALID_ARG before anything is launched (an
 *    address found usable once is not asked about again on that thread, so
 *    a buffer freed and its address reused for another kind of memory slips
 *    through).  Buffer sizes cannot be checked this way: they must be at
 *    least what each call states.
 *  - bf16 tensors are passed as void* holding IEEE bfloat16 bits.
 *  - Device pointers of row data (x, recv, expert_out, out) must be 16-byte
 *    aligned; hidden must be a multiple of 8 (rows are whole 16-byte units).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream)
 *    of the handle's device.  A call on a handle makes that device current
 *    while it runs and then restores the caller's current device.
 *    Work is enqueued on it and the call returns without waiting, except where
 *    a call says it synchronises.
 *  - Every call returns an ep_status.  Arguments are checked on the host before
 *    anything is launched (EP_ERR_INVALID_ARG).  Errors found on the device
 *    (a pick outside [-1, E), a receive buffer too small, a bounded wait that
 *    ran out) set a sticky per-handle error word; the kernels then stop early
 *    and never trap.  Read it with ep_last_device_status; clear it (and the
 *    ring state) with ep_reset.
 *  - A handle is used by one host thread at a time; calls on one handle must
 *    be ordered on one stream (they share the handle's rings and scratch).
 */
#ifndef EP_H_
#define EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  EP_ERR_CAPACITY is the analogue of GIN_ERR_WINDOW_FULL and
 * EP_ERR_NOT_READY of GIN_ERR_SIGNAL_PENDING ([GIN] s4.2.1 error codes). */
typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,
    EP_ERR_CAPACITY = 2,
    EP_ERR_TIMEOUT = 3,
    EP_ERR_CUDA = 4,
    EP_ERR_NOT_READY = 5
} ep_status;

typedef struct ep_ctx *ep_handle;

/* Layer shape and ring settings.  Defaults (ep_config_init) are the
 * [UCCL-EP] s5.2 tuning table: 8 channels (HT_CHANNELS), ring depth 1024
 * (FIFO_DEPTH), 256 commands in flight per channel (MAX_INFLIGHT), consumer
 * poll batch 32 (DRAIN_BATCH_SIZE); batches of up to 8 commands (s2.2); rows
 * per message 8 when a row is under 7 KB, else 1 (s4.1, s5.3). */
typedef struct {
    int32_t num_ranks;       /* R, 1..64 */
    int32_t tokens_per_rank; /* Tpr >= 1; T = R * Tpr tokens, source rank of t is t / Tpr */
    int32_t hidden;          /* H, multiple of 8; a row is 2*H bytes of bf16 */
    int32_t num_experts;     /* E, a multiple of R; expert e lives on rank e / (E/R) */
    int32_t topk;            /* K, 1..32 */
    int32_t channels;        /* C, 1..64: rings; a message to rank d goes to ring d % C.
                                The default is the tuning table's 8; a small layer's
                                posting tail shrinks with more rings (the 32-rank,
                                128-token layer: 108.6 us at 8, 100.7 at 16) */
    int32_t ring_depth;      /* D, power of two, 8..8192 slots per ring */
    int32_t max_inflight;    /* 8..D: producers wait while head - tail would exceed it */
    int32_t batch;           /* 1..8 commands reserved per head update */
    int32_t rows_per_msg;    /* G >= 1 rows per TransferCmd message; 0 = default rule */
    int32_t drain_batch;     /* 32 or a multiple of it: slots a consumer polls per step */
    int32_t debug_flags;     /* EP_DEBUG_* bits; 0 in normal use */
    int32_t num_sms;         /* SMs the dispatch and combine grids may occupy, leaving
                                the rest to concurrent work; 0 = all.  The dispatch
                                needs at least channels + 1 */
    int32_t reserved;        /* 0 */
    uint64_t timeout_ns;     /* limit of every device-side wait; 0 = 2 s */
} ep_config;

/* Test hook: ring consumers do not run, so producers see a full ring and their
 * bounded flow-control wait ends in EP_ERR_TIMEOUT (no GPU hang, no trap). */
#define EP_DEBUG_DISABLE_CONSUMER 0x1
/* Test hook: the per-message landed-row counters of multi-row messages
 * (rows_per_msg > 1) live in device memory even where a ring's counters fit in
 * its shared memory -- the path taken when a ring's messages outnumber that
 * room.  Results are unchanged. */
#define EP_DEBUG_DEVICE_COUNTERS 0x2

/* One ring record ([UCCL-EP] s2.3 TransferCmd; WRITE only), 32 bytes.
 *  dst_rank:   destination rank d.
 *  size:       payload bytes = rows * 2 * hidden.
 *  src_offset: byte offset into the logical send buffer, whose rows are
 *              ordered (source rank, destination rank, row) -- send_off.
 *  dst_offset: byte offset into rank d's receive window, i.e. relative to
 *              recv row recv_base[d] ([GIN] s2.2.1 byte-offset windows).
 *  type:       0 = WRITE.  reserved: 0. */
typedef struct {
    uint32_t dst_rank;
    uint32_t size;
    uint64_t src_offset;
    uint64_t dst_offset;
    uint32_t type;
    uint32_t reserved;
} ep_transfer_cmd;

/* Caller-owned device outputs of ep_layout (inputs of dispatch / combine).
 * Shapes use R ranks, T tokens, E experts; all int32 except is_token_in_rank.
 *  num_tokens_per_expert [R, E]: picks of rank s's tokens that name expert e
 *  num_tokens_per_rank   [R, R]: cnt[s][d] = tokens of rank s that reach rank d
 *  is_token_in_rank      [T, R] uint8: 1 if some pick of t lives on rank d
 *  token_slot            [T, R]: row of (t, d) inside rank d's window, or -1
 *  recv_off              [R, R]: first window row of source s in window d
 *  send_off              [R, R]: row-major exclusive scan of cnt
 *  msg_count             [R, R]: ceil(cnt / G)
 *  recv_count            [R]:    rows received by rank d
 *  recv_base             [R]:    exclusive scan of recv_count (window starts)
 *  expert_off            [E]:    exclusive scan over e of total picks of e */
typedef struct {
    int32_t *num_tokens_per_expert;
    int32_t *num_tokens_per_rank;
    uint8_t *is_token_in_rank;
    int32_t *token_slot;
    int32_t *recv_off;
    int32_t *send_off;
    int32_t *msg_count;
    int32_t *recv_count;
    int32_t *recv_base;
    int32_t *expert_off;
} ep_layout_out;

/* Caller-owned device outputs of ep_expert_layout: the expert-major view of
 * the receive buffer that a rank's grouped expert step consumes.  N receive
 * rows, K picks per token, E experts, Er = E / R experts per rank.
 *  recv_topk_idx     [N, K] int32: pick k of the row's token as a local
 *                    expert id (e - d*Er) if it lives on the row's rank d,
 *                    else -1
 *  recv_topk_weights [N, K] fp32:  topk_weights[t][k] where recv_topk_idx is
 *                    not -1, else 0
 *  recv_src_token    [N] int32:    the token t the row was copied from
 *  expert_rows       [M] int32:    receive rows grouped by expert: expert e's
 *                    rows are expert_rows[expert_off[e] + j], j <
 *                    expert_count[e], in increasing row (= token) order;
 *                    M = number of picks that are not -1 (at most T*K)
 *  expert_count      [E] int32:    picks of expert e over all source ranks */
typedef struct {
    int32_t *recv_topk_idx;
    float *recv_topk_weights;
    int32_t *recv_src_token;
    int32_t *expert_rows;
    int32_t *expert_count;
} ep_expert_layout_out;

/* Library-owned view of the per-channel TransferCmd logs written by the ring
 * consumers during the last ep_dispatch.  Device pointers, valid until
 * ep_destroy; channel c's records are cmds[c * capacity_per_channel + i]
 * for i < count[c] (count is a device array of int64, written at the end of
 * each dispatch). */
typedef struct {
    ep_transfer_cmd *cmds;
    int64_t *count;
    int64_t capacity_per_channel;
    int32_t channels;
} ep_cmd_log;

/* Per-channel ring counters, copied to the host by ep_ring_stats_get.
 * head/tail are cumulative since create/reset; the rest as named. */
typedef struct {
    uint64_t head;           /* commands reserved (producers) */
    uint64_t tail;           /* commands retired (consumer) */
    uint64_t batches;        /* head reservations (batch pushes) */
    uint64_t stall_polls;    /* producer polls that found the ring too full */
    uint32_t max_batch;      /* largest batch pushed */
    uint32_t max_inflight;   /* largest head - tail a producer observed after reserving */
    int64_t last_count;      /* commands retired by the last dispatch */
} ep_ring_stats;

/* Derived launch parameters of a handle (for reports and tests). */
typedef struct {
    int32_t rows_per_msg;         /* G in use */
    int32_t sm_count;             /* SMs of the device */
    int32_t dispatch_grid;        /* CTAs of the persistent dispatch kernel */
    int32_t dispatch_stages;      /* shared-memory row stages per dispatch CTA */
    int32_t dispatch_stage_bytes; /* bytes per stage */
    int32_t combine_grid;         /* CTAs of the combine kernel */
    int32_t layout_tiles;         /* token tiles of the layout scan */
    int32_t dispatch_chunk_tokens; /* tokens per dispatch chunk: 32, halved down to 4
                                      while the layer has < 4 chunks per copy CTA */
    int64_t log_capacity_per_channel;
    int64_t scratch_bytes;        /* device memory the handle allocated */
} ep_info;

/* Fill *cfg with the shape and the [UCCL-EP] s5.2 defaults.  Host only. */
ep_status ep_config_init(ep_config *cfg, int32_t num_ranks, int32_t tokens_per_rank,
                         int32_t hidden, int32_t num_experts, int32_t topk);

/* Check *cfg without touching the GPU.  Host only. */
ep_status ep_config_check(const ep_config *cfg);

/* Create a handle on the current device: allocates the rings, their logs and
 * the layout scratch (cudaMalloc), sized from *cfg.  Synchronous. */
ep_status ep_create(const ep_config *cfg, ep_handle *out);

/* Free everything ep_create allocated.  Synchronises the device first. */
ep_status ep_destroy(ep_handle h);

/* Static string for a status code. */
const char *ep_status_str(ep_status s);

/* Synchronise the device and read the sticky device error word into *code
 * (EP_OK if none).  Returns EP_OK unless the read itself failed. */
ep_status ep_last_device_status(ep_handle h, int32_t *code);

/* Synchronise the device, then clear the error word, the rings (head, tail,
 * slots, statistics) and the layout scan state. */
ep_status ep_reset(ep_handle h);

/* ep_layout -- token layout of one EP layer ([UCCL-EP] s1: EP needs
 * fine-grained token-level communication; [NOTES] names a layout/rank mismatch
 * as an EP failure class).  One single-pass kernel: a warp-aggregated
 * histogram of picks per (source rank, expert), rank membership per token,
 * and a decoupled-lookback scan down each destination column giving
 * token_slot; the last tile to finish derives the small scans.
 *  topk_idx: device int32 [T, K]; -1 = no pick; other values outside [0, E)
 *            set EP_ERR_INVALID_ARG on the device and are skipped.
 *  out:      caller-owned device outputs (all ten pointers required).
 *  n_recv_host: if non-NULL, the call synchronises `stream` and writes
 *            N = sum(recv_count), so the caller can size the receive buffer;
 *            if NULL the call is fully asynchronous. */
ep_status ep_layout(ep_handle h, const int32_t *topk_idx, const ep_layout_out *out,
                    int64_t *n_recv_host, void *stream);

/* ep_dispatch -- send every token row to each destination rank it reaches,
 * once per rank ([UCCL-EP] s6 "Dispatch"; s4.1 pipelined DispatchKernel), and
 * post one TransferCmd per message of up to G rows into ring d % C in batches
 * of up to `batch` commands, with producers waiting while a ring holds
 * max_inflight commands ([UCCL-EP] s2.2 lock-free ring, batch enqueue, flow
 * control; s4.2 channels).  Consumer warps on the device retire each ring into
 * its log (ep_cmd_log) and advance its tail; the kernel ends when every ring
 * is drained ([UCCL-EP] s3.1 Drain).  One persistent cooperative kernel; rows
 * move through shared memory, each source row read once: TMA bulk loads, then
 * TMA bulk stores (rows over 4 KB) or vector stores from seven store warps
 * (rows of at most 4 KB).
 *  x:      device bf16 [T, H].
 *  layout: outputs of ep_layout for this routing (read on the device).
 *  recv:   device bf16 [recv_capacity_rows, H]; rows [0, N) are written.
 *          If N > recv_capacity_rows the device sets EP_ERR_CAPACITY and
 *          nothing is written. */
ep_status ep_dispatch(ep_handle h, const void *x, const ep_layout_out *layout, void *recv,
                      int64_t recv_capacity_rows, void *stream);

/* ep_combine -- top-k weighted reduction back to token order ([UCCL-EP] s6
 * "Combine"):
 *   out[t] = bf16_rne( acc ), acc = +0.0f; for k = 0..K-1 with a pick:
 *            acc = fmaf(topk_weights[t][k], expert_out[recv_base[d] + token_slot[t][d]], acc),
 *            d = topk_idx[t][k] / (E/R)
 * in fp32, in that fixed order.
 *  expert_out: device bf16 [expert_out_rows, H] (one row per receive row).
 *  topk_weights: device fp32 [T, K]; topk_idx: device int32 [T, K].
 *  out: device bf16 [T, H].  A row index outside [0, expert_out_rows) sets
 *  EP_ERR_INVALID_ARG on the device and that pick is skipped. */
ep_status ep_combine(ep_handle h, const void *expert_out, int64_t expert_out_rows,
                     const float *topk_weights, const int32_t *topk_idx,
                     const ep_layout_out *layout, void *out, void *stream);

/* Pieces of one layer, for overlap: the layer split into micro-batches so
 * that the expert work on one piece, or the next layer, runs while another
 * piece moves ([GIN] s3.1.2 expert computation overlapping communication; the
 * GPU communication notes' "communication and compute overlap": combine
 * overlapped with the next layer, fixed launch order in CUDA graphs).  With
 * ep_config.num_sms below the SM count the dispatch and combine grids leave
 * the remaining SMs to concurrent kernels.
 *
 * ep_dispatch_ranks -- ep_dispatch restricted to the tokens of source ranks
 * [src_begin, src_end): their rows are copied to their receive rows, and the
 * TransferCmds (and arrival signals) of the pairs (s, d) with s in the range
 * are posted; other receive rows are not written.  The log then holds this
 * call's commands.  Pieces that together cover [0, R) leave recv, the logged
 * command multiset and the signals as one ep_dispatch does.  Calls on one
 * handle must not overlap each other (they share the rings).
 * 0 <= src_begin <= src_end <= R, else EP_ERR_INVALID_ARG. */
ep_status ep_dispatch_ranks(ep_handle h, const void *x, const ep_layout_out *layout, void *recv,
                            int64_t recv_capacity_rows, int32_t src_begin, int32_t src_end, void *stream);

/* ep_combine_tokens -- ep_combine for tokens [t_begin, t_end) only: rows
 * t_begin .. t_end-1 of out (still [T, H]) are written.
 * 0 <= t_begin <= t_end <= T, else EP_ERR_INVALID_ARG. */
ep_status ep_combine_tokens(ep_handle h, const void *expert_out, int64_t expert_out_rows,
                            const float *topk_weights, const int32_t *topk_idx,
                            const ep_layout_out *layout, void *out, int64_t t_begin, int64_t t_end,
                            void *stream);

/* ep_expert_layout -- expert-major receive metadata ([UCCL-EP] s1: each
 * token goes to the experts of its top-k picks, and the receiving rank runs
 * those experts on the rows it received).  Needs only the layout, not the
 * dispatched rows, so it may run on another stream while ep_dispatch moves
 * the data.  One single-pass kernel over tiles of 256 tokens (128 when
 * E > 2048): per tile a bitmask of tokens per expert in shared memory, a
 * decoupled-lookback scan down each expert column giving each pick's position
 * in its expert's segment, and the per-row metadata written from the token's
 * own picks.
 *  topk_idx, topk_weights: device int32 / fp32 [T, K], the inputs of
 *            ep_layout and ep_combine.  A pick outside [-1, E), or a token
 *            naming one expert twice, sets EP_ERR_INVALID_ARG on the device
 *            and that pick is skipped.
 *  layout:   ep_layout's outputs for this routing (token_slot, recv_base and
 *            expert_off are read on the device).
 *  out:      caller-owned device outputs (all five pointers required).
 *  recv_rows: rows of recv_topk_idx / recv_topk_weights / recv_src_token
 *            (at least N); expert_rows_capacity: entries of expert_rows (at
 *            least M; T*K always suffices).  A row or an entry beyond them
 *            sets EP_ERR_CAPACITY on the device and is not written.
 * The handle's scratch for this call (the lookback descriptors) grows as
 * T*E/32 bytes, T*E/16 when E > 2048. */
ep_status ep_expert_layout(ep_handle h, const int32_t *topk_idx, const float *topk_weights,
                           const ep_layout_out *layout, const ep_expert_layout_out *out,
                           int64_t recv_rows, int64_t expert_rows_capacity, void *stream);

/* Arrival signals, one per destination rank ([GIN] s2.2.2 completion
 * notification: remote-completion signals bumped by atomic adds, addressed by
 * id; s2.1.2 put with SignalInc, then waitSignal on an expected value).
 * signal[d] counts the messages of every ep_dispatch since ep_create,
 * ep_reset or ep_signal_reset whose rows have landed in rank d's window; one
 * dispatch adds sum_s msg_count[s][d].  Each increment is a GPU-scope release
 * made after the message's rows were written.  include/ep_signal.cuh has the
 * device-side read and bounded wait for a consumer's own kernels. */

/* Device address of signal[R] (uint64), valid until ep_destroy. */
ep_status ep_signal_ptr(ep_handle h, const uint64_t **signals);

/* Copy signal[0, n) to host array out[n] (synchronises the device); n must
 * not exceed the rank count. */
ep_status ep_signal_get(ep_handle h, uint64_t *host_out, int32_t n);

/* Zero every signal, ordered on `stream` ([GIN] s4.2.1: reset a signal
 * before reuse). */
ep_status ep_signal_reset(ep_handle h, void *stream);

/* Enqueue on `stream` a one-thread kernel that polls signal[dst_rank] (acquire
 * reads, 100 ns back-off) until it reaches `expected` or timeout_ns (at most
 * 10 s) has passed, then writes EP_OK or EP_ERR_NOT_READY (the analogue of
 * GIN_ERR_SIGNAL_PENDING) to the device int32 *status_out.  The handle's
 * error word is not touched.  Wait for a dispatch enqueued before it (on this
 * stream or ordered by an event): a wait running while the dispatch it waits
 * for has not started can hold the SMs the dispatch needs, and then it runs
 * out.  dst_rank outside [0, R) returns EP_ERR_INVALID_ARG. */
ep_status ep_wait_signal(ep_handle h, int32_t dst_rank, uint64_t expected, uint64_t timeout_ns,
                         int32_t *status_out, void *stream);

/* Device pointers of the TransferCmd logs (no synchronisation). */
ep_status ep_cmd_log_get(ep_handle h, ep_cmd_log *out);

/* Copy the ring counters of channels [0, n) to host array out[n]
 * (synchronises the device).  n must not exceed the channel count. */
ep_status ep_ring_stats_get(ep_handle h, ep_ring_stats *out, int32_t n);

/* Completion query ([UCCL-EP] s2.2 CheckCompletion): EP_OK if command index
 * cmd_idx (cumulative since create/reset) of `channel` has been retired by its
 * consumer -- the channel's tail has passed it -- EP_ERR_NOT_READY if not yet.
 * Synchronises the device, then reads the tail. */
ep_status ep_check_completion(ep_handle h, int32_t channel, uint64_t cmd_idx);

/* Launch parameters and allocation size of a handle.  Host only. */
ep_status ep_get_info(ep_handle h, ep_info *out);

/* ep_layout_static -- ep_layout for callers that cannot allocate device
 * memory.  The articles have no counterpart: this is a service of this
 * library.  Some callers cannot call cudaMalloc, and so cannot create a
 * handle: cudaMalloc may synchronise the whole device, which a serving loop
 * that must never stall cannot afford, and a framework whose caching
 * allocator owns all device memory may forbid allocations made behind its
 * back.  This call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine) and needs no handle: the layout's scratch lives
 * in one fixed device array built into the library, about 785 KB, which every
 * GPU that loads the library holds until the process exits.
 *  cfg:         the layer's shape (ep_config_check rules); only num_ranks,
 *               tokens_per_rank, hidden, num_experts, topk and rows_per_msg
 *               matter here.  Sizes beyond the array's capacity -- more than
 *               262144 tokens (num_ranks * tokens_per_rank), 64 ranks or 1024
 *               experts -- return EP_ERR_CAPACITY and launch nothing.
 *  topk_idx, out: as for ep_layout (caller-owned device memory); the outputs
 *               are the ones ep_layout writes.
 *  n_recv_host: if non-NULL, the call synchronises `stream`, writes N and
 *               returns the device-side status of this call (EP_ERR_INVALID_ARG
 *               for a pick outside [-1, E)); if NULL it returns without waiting
 *               and device-side errors are not reported: the next call clears
 *               the array's error word before it starts, so a caller that
 *               never waits for N must validate topk_idx itself (every pick in
 *               [-1, E)) or check the outputs by other means.
 * The first call on a device looks up the array's device address (once per
 * device, under a lock) and keeps it for the life of the process; make that
 * first call before any stream capture.  cudaDeviceReset on a device after
 * its first call is not supported: the address kept would then be stale.
 * Every call on a device shares the one array and the call clears the parts
 * it needs at zero first, so calls must not overlap on the GPU: two calls in
 * flight at once (on different streams, or from different threads) race. */
ep_status ep_layout_static(const ep_config *cfg, const int32_t *topk_idx, const ep_layout_out *out,
                           int64_t *n_recv_host, void *stream);

/* SM partitions for overlapping the layer's data movement with computation
 * (GPU communication notes, communication/computation overlap: DeepEP gives
 * its dispatch and combine kernels a fixed SM budget and the rest of the GPU
 * to the expert GEMMs).  ep_sm_split_create divides device `device`'s SMs into
 * two disjoint partitions with the driver's green contexts: at least
 * compute_sms SMs (rounded up to the device's partition granularity, 8 SMs
 * on this architecture) for computation and the remainder for communication,
 * each with a non-blocking stream whose work runs only on its partition.  The
 * streams belong to the device's primary context, so device memory, events
 * and every other stream work with them as usual.  To overlap, run
 * ep_layout/ep_dispatch/ep_combine on the communication stream of a handle
 * made with num_sms = the communication partition's SM count (a cooperative
 * dispatch must fit in its partition), the caller's compute on the compute
 * stream, and order the two with events only: no kernel on one stream may
 * wait on the other's progress (partitions do not guarantee that both run at
 * once).  compute_sms must leave SMs for communication, else
 * EP_ERR_INVALID_ARG; driver failures are EP_ERR_CUDA.  The caller owns the
 * split and frees it with ep_sm_split_destroy after the work queued on its
 * streams (destroy waits for both streams first). */
typedef struct ep_sm_split_s *ep_sm_split;
ep_status ep_sm_split_create(int32_t device, int32_t compute_sms, ep_sm_split *out);
/* The partitions' streams (cudaStream_t) and SM counts; any output may be NULL. */
ep_status ep_sm_split_get(ep_sm_split split, void **comm_stream, int32_t *comm_sms, void **compute_stream,
                          int32_t *compute_sms);
ep_status ep_sm_split_destroy(ep_sm_split split);
/* Diagnostic: enqueue on `stream` `blocks` (1..2^20) one-warp blocks that each
 * run about 2 us and write the id of the SM they ran on to sm_ids_out[block]
 * (caller-owned device int32 array).  Shows which SMs a stream's work may
 * use. */
ep_status ep_sm_ids(void *stream, int32_t blocks, int32_t *sm_ids_out);

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */
