// ep_combine.cu -- top-k weighted reduction of expert outputs back to token
// order (UCCL-EP article s6 "Combine"), sm_103a.
//
//   out[t] = bf16_rne(acc), acc = +0.0f, then for k = 0..K-1 with a pick:
//            acc = fmaf(w[t][k], expert_out[recv_base[d] + token_slot[t][d]], acc),
//            d = topk_idx[t][k] / (E/R)
//
// One warp per token.  Lane k < K resolves pick k to its receive row; the rows
// and weights are broadcast with shuffles; then each lane walks the row in
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

template <int KMAX, int SEGS>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kCombineThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kCombineThreads) >> 5;
    const int K = p.K, R = p.R;
    const int64_t B = p.row_bytes;

    for (int64_t t = p.t_begin + warp0; t < p.t_end; t += nwarps) {
        int64_t row = -1;
        float w = 0.0f;
        if (lane < K) {
            const int e = __ldg(p.topk_idx + t * K + lane);
            if (e >= 0 && e < p.E) {
                const int d = e / p.Er;
                const int slot = __ldg(p.token_slot + t * R + d);
                const int64_t r = static_cast<int64_t>(__ldg(p.recv_base + d)) + slot;
                if (slot >= 0 && r >= 0 && r < p.eo_rows) {
                    row = r;
                    w = __ldg(p.w + t * K + lane);
                } else {
                    set_error(p.dev.err, EP_ERR_INVALID_ARG);
                }
            } else if (e != -1) {
                set_error(p.dev.err, EP_ERR_INVALID_ARG);
            }
        }
        const uint8_t *src[KMAX];
        float wk[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int64_t r = __shfl_sync(0xffffffffu, row, k);
            wk[k] = __shfl_sync(0xffffffffu, w, k);
            src[k] = (k < K && r >= 0) ? p.expert_out + r * B : nullptr;
        }
        uint8_t *dst = p.out + t * B;
        for (int s0 = lane; s0 < p.nseg; s0 += 32 * SEGS) {
            uint4 v[SEGS][KMAX];
#pragma unroll
            for (int j = 0; j < SEGS; ++j) {
                const int seg = s0 + 32 * j;
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    v[j][k] = make_uint4(0u, 0u, 0u, 0u);
                    if (seg < p.nseg && src[k] != nullptr)
                        v[j][k] = __ldg(reinterpret_cast<const uint4 *>(src[k] + static_cast<int64_t>(seg) * 16));
                }
            }
#pragma unroll
            for (int j = 0; j < SEGS; ++j) {
                const int seg = s0 + 32 * j;
                if (seg >= p.nseg) break;
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
    }
}

template <int KMAX, int SEGS>
ep_status launch_k(ep_ctx *h, const CombineParams &p, cudaStream_t st) {
    // one warp per token, at most the planned grid (grid-stride beyond it)
    const int64_t warps_per_cta = kCombineThreads / 32;
    const int64_t need = (p.t_end - p.t_begin + warps_per_cta - 1) / warps_per_cta;
    const int grid = static_cast<int>(need < h->comb_grid ? need : h->comb_grid);
    if (grid <= 0) return EP_OK;
    combine_kernel<KMAX, SEGS><<<grid, kCombineThreads, 0, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace

ep_status plan_combine(ep_ctx *h) {
    const int64_t T = static_cast<int64_t>(h->cfg.num_ranks) * h->cfg.tokens_per_rank;
    const int64_t warps_per_cta = kCombineThreads / 32;
    const int64_t need = (T + warps_per_cta - 1) / warps_per_cta;
    const int64_t sms = h->cfg.num_sms > 0 && h->cfg.num_sms < h->sm_count ? h->cfg.num_sms : h->sm_count;
    const int64_t cap = sms * 32;   // grid-stride beyond this
    h->comb_grid = static_cast<int>(need < cap ? need : cap);
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
