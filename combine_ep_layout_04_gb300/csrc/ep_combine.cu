// ep_combine.cu -- top-k weighted reduction of expert outputs back to token
// order (UCCL-EP article s6 "Combine"), sm_103a.
//
//   out[t] = bf16_rne(acc), acc = +0.0f, then for k = 0..K-1 with a pick:
//            acc = fmaf(w[t][k], expert_out[recv_base[d] + token_slot[t][d]], acc),
//            d = topk_idx[t][k] / (E/R)
//
// One warp per token (or per part of a token's row when the layer is small).
// Lane k < K resolves pick k to its receive row; the rows and weights are
// broadcast with shuffles; then each lane walks the row in
// 16-byte segments, issuing the loads of all K rows for SEGS segments before
// the first multiply-add so that SEGS*K loads are in flight per lane.  Picks
// that share a rank read the same row: the second read is served by L1, so
// each distinct row crosses HBM once.  The fp32 chain runs in the fixed order
// k = 0..K-1 with fused multiply-adds, then rounds to bf16 (nearest, even).
// This is HBM-bound data movement: no tensor cores are involved.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kCombineThreads = 256;
constexpr int64_t kBigRowBytes = 8192;

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4 &v) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w, __uint_as_float(u[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

// Lane k < K turns pick e of token t into its receive row and weight
// (row -1: no pick); other lanes return row -1.
__device__ __forceinline__ void resolve_pick(const CombineParams &p, int64_t t, int lane, int e, int64_t &row,
                                             float &w) {
    row = -1;
    w = 0.0f;
    if (lane >= p.K || t < 0) return;
    if (e >= 0 && e < p.E) {
        const int d = e / p.Er;
        const int slot = __ldg(p.token_slot + t * p.R + d);
        const int64_t r = static_cast<int64_t>(__ldg(p.recv_base + d)) + slot;
        if (slot >= 0 && r >= 0 && r < p.eo_rows) {
            row = r;
            w = __ldg(p.w + t * p.K + lane);
        } else {
            set_error(p.dev.err, EP_ERR_INVALID_ARG);
        }
    } else if (e != -1) {
        set_error(p.dev.err, EP_ERR_INVALID_ARG);
    }
}

// Work item i of a call: token t_begin + i / nparts, segments of part
// i % nparts.  Warps stride over the items.  Each warp loads the next item's
// picks before working on the current one and turns them into rows while the
// current item's loads are in flight, so an item waits on one round trip for
// its metadata, not three.
template <int KMAX, int SEGS>
__global__ void __launch_bounds__(kCombineThreads, KMAX <= 8 ? 2 : 1) combine_kernel(const CombineParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kCombineThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kCombineThreads) >> 5;
    const int K = p.K;
    const int64_t B = p.row_bytes;
    const int64_t items = (p.t_end - p.t_begin) * p.nparts;
    const int part_segs = (p.nseg + p.nparts - 1) / p.nparts;

    auto token_of = [&](int64_t it) -> int64_t { return it < items ? p.t_begin + it / p.nparts : -1; };
    int64_t item = warp0;
    int64_t row = -1;
    float w = 0.0f;
    {
        const int64_t t = token_of(item);
        const int e = (t >= 0 && lane < K) ? __ldg(p.topk_idx + t * K + lane) : -1;
        resolve_pick(p, t, lane, e, row, w);
    }
    for (; item < items; item += nwarps) {
        const int64_t t = p.t_begin + item / p.nparts;
        const int part = static_cast<int>(item % p.nparts);
        const int64_t t_next = token_of(item + nwarps);
        const int e_next = (t_next >= 0 && lane < K) ? __ldg(p.topk_idx + t_next * K + lane) : -1;
        const uint8_t *src[KMAX];
        float wk[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int64_t r = __shfl_sync(0xffffffffu, row, k);
            wk[k] = __shfl_sync(0xffffffffu, w, k);
            src[k] = (k < K && r >= 0) ? p.expert_out + r * B : nullptr;
        }
        uint8_t *dst = p.out + t * B;
        const int seg_lo = part * part_segs, seg_hi = min(p.nseg, seg_lo + part_segs);
        bool resolved = false;
        for (int s0 = seg_lo + lane; s0 < seg_hi; s0 += 32 * SEGS) {
            uint4 v[SEGS][KMAX];
#pragma unroll
            for (int j = 0; j < SEGS; ++j) {
                const int seg = s0 + 32 * j;
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    v[j][k] = make_uint4(0u, 0u, 0u, 0u);
                    if (seg < seg_hi && src[k] != nullptr)
                        v[j][k] = __ldg(reinterpret_cast<const uint4 *>(src[k] + static_cast<int64_t>(seg) * 16));
                }
            }
            if (!resolved) {   // the next item's rows, while these loads fly
                resolve_pick(p, t_next, lane, e_next, row, w);
                resolved = true;
            }
#pragma unroll
            for (int j = 0; j < SEGS; ++j) {
                const int seg = s0 + 32 * j;
                if (seg >= seg_hi) break;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
                for (int k = 0; k < KMAX; ++k)
                    if (src[k] != nullptr) fma8(acc, wk[k], v[j][k]);
                uint4 o;
                o.x = pack_bf16x2(acc[0], acc[1]);
                o.y = pack_bf16x2(acc[2], acc[3]);
                o.z = pack_bf16x2(acc[4], acc[5]);
                o.w = pack_bf16x2(acc[6], acc[7]);
                *reinterpret_cast<uint4 *>(dst + static_cast<int64_t>(seg) * 16) = o;
            }
        }
        if (!resolved) resolve_pick(p, t_next, lane, e_next, row, w);
    }
}

template <int KMAX, int SEGS>
ep_status launch_k(ep_ctx *h, CombineParams &p, cudaStream_t st) {
    // Rows of 8 KB and more: one item per token and up to 16 resident
    // grids' worth of CTAs (the block scheduler keeps every SM fed).  Smaller
    // rows: the resident grid, warps striding over the items, and each
    // token's row split into parts when there are too few tokens to give
    // every warp several items.  (Measured: the first is faster for 14 KB
    // rows, the second for 2-4 KB rows.)
    const int64_t ntok = p.t_end - p.t_begin;
    if (ntok <= 0) return EP_OK;
    const int64_t warps_per_cta = kCombineThreads / 32;
    const int64_t resident_warps = static_cast<int64_t>(h->comb_grid) * warps_per_cta;
    const bool big_rows = p.row_bytes >= kBigRowBytes;
    p.nparts = 1;
    while (!big_rows && p.nparts < 8 && ntok * p.nparts < 4 * resident_warps &&
           p.nseg / (2 * p.nparts) >= 32 * SEGS)
        p.nparts *= 2;
    const int64_t need = (ntok * p.nparts + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = big_rows ? 16ll * h->comb_grid : h->comb_grid;
    const int grid = static_cast<int>(need < cap ? need : cap);
    combine_kernel<KMAX, SEGS><<<grid, kCombineThreads, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

template <int KMAX, int SEGS>
int resident_ctas_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel<KMAX, SEGS>, kCombineThreads, 0) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace

ep_status plan_combine(ep_ctx *h) {
    // the resident grid of the kernel this handle's K selects, on the SMs
    // the handle may use
    const int K = h->cfg.topk;
    const int per_sm = K <= 2 ? resident_ctas_per_sm<2, 4>() : K <= 4 ? resident_ctas_per_sm<4, 4>()
                     : K <= 8 ? resident_ctas_per_sm<8, 2>() : K <= 16 ? resident_ctas_per_sm<16, 1>()
                     : resident_ctas_per_sm<32, 1>();
    if (per_sm < 1) return EP_ERR_CUDA;
    const int sms = h->cfg.num_sms > 0 && h->cfg.num_sms < h->sm_count ? h->cfg.num_sms : h->sm_count;
    h->comb_grid = per_sm * sms;
    h->comb_threads = kCombineThreads;
    return EP_OK;
}

ep_status launch_combine(ep_ctx *h, const void *expert_out, int64_t eo_rows, const float *w,
                         const int32_t *topk_idx, const ep_layout_out *lay, void *out, int64_t t_begin,
                         int64_t t_end, cudaStream_t st) {
    CombineParams p{};
    p.expert_out = static_cast<const uint8_t *>(expert_out);
    p.eo_rows = eo_rows;
    p.w = w;
    p.topk_idx = topk_idx;
    p.token_slot = lay->token_slot;
    p.recv_base = lay->recv_base;
    p.out = static_cast<uint8_t *>(out);
    p.dev = h->dev;
    p.R = h->cfg.num_ranks;
    p.T = static_cast<int64_t>(p.R) * h->cfg.tokens_per_rank;
    p.t_begin = t_begin;
    p.t_end = t_end;
    p.K = h->cfg.topk;
    p.E = h->cfg.num_experts;
    p.Er = p.E / p.R;
    p.row_bytes = 2ll * h->cfg.hidden;
    p.nseg = h->cfg.hidden / 8;
    const int K = p.K;
    if (K <= 2) return launch_k<2, 4>(h, p, st);
    if (K <= 4) return launch_k<4, 4>(h, p, st);
    if (K <= 8) return launch_k<8, 2>(h, p, st);
    if (K <= 16) return launch_k<16, 1>(h, p, st);
    return launch_k<32, 1>(h, p, st);
}

}  // namespace ep
