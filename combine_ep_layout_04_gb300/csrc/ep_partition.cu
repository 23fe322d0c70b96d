// ep_partition.cu -- disjoint SM partitions for overlapping the layer's data
// movement with computation (the GPU communication notes' overlap of MoE
// dispatch/combine with compute; DeepEP gives its communication kernels a
// fixed SM budget and the rest to the GEMMs).
//
// The split is made with the driver's green contexts: the device's SM
// resource is divided into a group of at least `compute_sms` SMs and the
// remainder, a green context is made on each, and each gets a non-blocking
// stream.  Work launched on a stream runs only on its partition's SMs; the
// streams belong to the device's primary context, so memory, events and the
// runtime API are shared with ordinary streams.  Driver entry points are
// looked up at run time through the runtime, so the library does not link
// libcuda.
#include <cuda.h>

#include "ep_internal.cuh"

struct ep_sm_split_s {
    int device;
    CUgreenCtx ctx[2];        // [0] communication, [1] compute
    CUstream stream[2];
    int sms[2];
};

namespace {

struct DriverFns {
    CUresult (*device_get)(CUdevice *, int);
    CUresult (*get_resource)(CUdevice, CUdevResource *, CUdevResourceType);
    CUresult (*split)(CUdevResource *, unsigned int *, const CUdevResource *, CUdevResource *, unsigned int,
                      unsigned int);
    CUresult (*gen_desc)(CUdevResourceDesc *, CUdevResource *, unsigned int);
    CUresult (*ctx_create)(CUgreenCtx *, CUdevResourceDesc, CUdevice, unsigned int);
    CUresult (*ctx_destroy)(CUgreenCtx);
    CUresult (*stream_create)(CUstream *, CUgreenCtx, unsigned int, int);
    CUresult (*stream_destroy)(CUstream);
    bool ok;
};

template <typename F>
bool lookup(const char *name, F *fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12080, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const DriverFns &driver() {
    static DriverFns d = [] {
        DriverFns f{};
        f.ok = lookup("cuDeviceGet", &f.device_get) && lookup("cuDeviceGetDevResource", &f.get_resource) &&
               lookup("cuDevSmResourceSplitByCount", &f.split) && lookup("cuDevResourceGenerateDesc", &f.gen_desc) &&
               lookup("cuGreenCtxCreate", &f.ctx_create) && lookup("cuGreenCtxDestroy", &f.ctx_destroy) &&
               lookup("cuGreenCtxStreamCreate", &f.stream_create) && lookup("cuStreamDestroy", &f.stream_destroy);
        return f;
    }();
    return d;
}

void release(const DriverFns &f, ep_sm_split_s *s) {
    for (int i = 0; i < 2; ++i) {
        if (s->stream[i]) f.stream_destroy(s->stream[i]);
        if (s->ctx[i]) f.ctx_destroy(s->ctx[i]);
    }
    delete s;
}

// One block per entry; each waits about 2 us (bounded by the global timer) so
// that the blocks spread over every SM the launch may use, then records the
// SM it ran on.
__global__ void sm_ids_kernel(int32_t *out) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const uint64_t t0 = ep::globaltimer_ns();
    while (ep::globaltimer_ns() - t0 < 2000) {
    }
    if (threadIdx.x == 0) out[blockIdx.x] = static_cast<int32_t>(smid);
}

}  // namespace

extern "C" {

ep_status ep_sm_split_create(int32_t device, int32_t compute_sms, ep_sm_split *out) {
    if (!out || device < 0 || compute_sms < 1) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return EP_ERR_CUDA;
    if (device >= ndev) return EP_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return EP_ERR_CUDA;
    // the primary context must be active before green contexts are made on it
    const bool init = cudaFree(nullptr) == cudaSuccess;
    cudaSetDevice(prev);
    if (!init) return EP_ERR_CUDA;
    const DriverFns &f = driver();
    if (!f.ok) return EP_ERR_CUDA;
    CUdevice dev;
    CUdevResource all{};
    if (f.device_get(&dev, device) != CUDA_SUCCESS || f.get_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS)
        return EP_ERR_CUDA;
    if (static_cast<unsigned>(compute_sms) >= all.sm.smCount) return EP_ERR_INVALID_ARG;
    CUdevResource grp{}, rest{};
    unsigned int ngroups = 1;
    if (f.split(&grp, &ngroups, &all, &rest, 0, static_cast<unsigned>(compute_sms)) != CUDA_SUCCESS || ngroups != 1 ||
        rest.sm.smCount == 0)
        return EP_ERR_INVALID_ARG;   // the partition granularity leaves no SMs for communication
    auto *s = new ep_sm_split_s{};
    s->device = device;
    CUdevResource *parts[2] = {&rest, &grp};
    for (int i = 0; i < 2; ++i) {
        CUdevResourceDesc desc;
        if (f.gen_desc(&desc, parts[i], 1) != CUDA_SUCCESS ||
            f.ctx_create(&s->ctx[i], desc, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS ||
            f.stream_create(&s->stream[i], s->ctx[i], CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
            release(f, s);
            return EP_ERR_CUDA;
        }
        s->sms[i] = static_cast<int>(parts[i]->sm.smCount);
    }
    *out = s;
    return EP_OK;
}

ep_status ep_sm_split_get(ep_sm_split s, void **comm_stream, int32_t *comm_sms, void **compute_stream,
                          int32_t *compute_sms) {
    if (!s) return EP_ERR_INVALID_ARG;
    if (comm_stream) *comm_stream = s->stream[0];
    if (comm_sms) *comm_sms = s->sms[0];
    if (compute_stream) *compute_stream = s->stream[1];
    if (compute_sms) *compute_sms = s->sms[1];
    return EP_OK;
}

ep_status ep_sm_split_destroy(ep_sm_split s) {
    if (!s) return EP_ERR_INVALID_ARG;
    const DriverFns &f = driver();
    if (!f.ok) return EP_ERR_CUDA;
    // work still queued on the partitions' streams finishes first
    for (int i = 0; i < 2; ++i)
        if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s->stream[i])) != cudaSuccess) return EP_ERR_CUDA;
    release(f, s);
    return EP_OK;
}

ep_status ep_sm_ids(void *stream, int32_t blocks, int32_t *sm_ids_out) {
    if (!sm_ids_out || blocks < 1 || blocks > (1 << 20)) return EP_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, sm_ids_out) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        return EP_ERR_INVALID_ARG;
    }
    sm_ids_kernel<<<blocks, 32, 0, static_cast<cudaStream_t>(stream)>>>(sm_ids_out);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // extern "C"
