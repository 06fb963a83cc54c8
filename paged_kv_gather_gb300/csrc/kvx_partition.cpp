// kvx_partition.cpp -- hard SM partitioning for I/O vs compute with green contexts.
//
// "Tutti: Making SSD-Backed KV Cache Practical for Long-Context LLM Serving", section 2
// Design 2, splits the GPU's SMs into a compute domain and an I/O domain with NVIDIA green
// contexts so that the I/O kernel never competes with compute for SMs.  Here the device's
// SM resource is split into `io_groups` I/O partitions of at least `io_sms` SMs each (the
// driver rounds up to its partition granularity) and a compute partition with the rest;
// each becomes a green context with one non-blocking stream.  Transfers launched on an
// I/O stream run only on that partition's SMs; anything launched on the compute stream (a
// GEMM, attention) runs only on the others.  Two I/O partitions keep a store and a load
// that run at once on fixed, disjoint SM sets.
//
// The driver entry points are looked up at run time through the CUDA runtime, so the
// library still loads on machines without a GPU driver.
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kvx_internal.h"

struct kvx_partition {
    static const int kMaxGroups = 8;
    int device = 0;
    int groups = 0;  // I/O groups; the compute partition is index `groups`
    CUgreenCtx ctx[kMaxGroups + 1] = {};
    CUstream stream[kMaxGroups + 1] = {};
    int sms[kMaxGroups + 1] = {};
};

namespace {

typedef CUresult (*PfnDeviceGet)(CUdevice *, int);
typedef CUresult (*PfnGetDevResource)(CUdevice, CUdevResource *, CUdevResourceType);
typedef CUresult (*PfnSplitByCount)(CUdevResource *, unsigned int *, const CUdevResource *,
                                    CUdevResource *, unsigned int, unsigned int);
typedef CUresult (*PfnGenerateDesc)(CUdevResourceDesc *, CUdevResource *, unsigned int);
typedef CUresult (*PfnGreenCtxCreate)(CUgreenCtx *, CUdevResourceDesc, CUdevice, unsigned int);
typedef CUresult (*PfnGreenCtxDestroy)(CUgreenCtx);
typedef CUresult (*PfnGreenCtxStreamCreate)(CUstream *, CUgreenCtx, unsigned int, int);
typedef CUresult (*PfnStreamDestroy)(CUstream);

struct Driver {
    PfnDeviceGet device_get = nullptr;
    PfnGetDevResource get_dev_resource = nullptr;
    PfnSplitByCount split_by_count = nullptr;
    PfnGenerateDesc generate_desc = nullptr;
    PfnGreenCtxCreate green_create = nullptr;
    PfnGreenCtxDestroy green_destroy = nullptr;
    PfnGreenCtxStreamCreate green_stream_create = nullptr;
    PfnStreamDestroy stream_destroy = nullptr;
};

template <class F>
bool entry(const char *name, F *fn)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &p, CUDART_VERSION, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
        cudaGetLastError();
        return false;
    }
    *fn = reinterpret_cast<F>(p);
    return true;
}

bool load_driver(Driver *d)
{
    return entry("cuDeviceGet", &d->device_get) &&
           entry("cuDeviceGetDevResource", &d->get_dev_resource) &&
           entry("cuDevSmResourceSplitByCount", &d->split_by_count) &&
           entry("cuDevResourceGenerateDesc", &d->generate_desc) &&
           entry("cuGreenCtxCreate", &d->green_create) &&
           entry("cuGreenCtxDestroy", &d->green_destroy) &&
           entry("cuGreenCtxStreamCreate", &d->green_stream_create) &&
           entry("cuStreamDestroy", &d->stream_destroy);
}

kvx_status fail(char *msg, size_t len, const char *fmt, ...)
{
    if (msg && len > 0) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(msg, len, fmt, ap);
        va_end(ap);
    }
    return KVX_ERR_CUDA;
}

void release(const Driver &d, kvx_partition *p)
{
    for (int g = 0; g <= kvx_partition::kMaxGroups; ++g) {
        if (p->stream[g])
            d.stream_destroy(p->stream[g]);
        if (p->ctx[g])
            d.green_destroy(p->ctx[g]);
        p->stream[g] = nullptr;
        p->ctx[g] = nullptr;
    }
}

}  // namespace

extern "C" {

kvx_status kvx_partition_create(int device, int io_groups, int io_sms, int io_priority,
                                int compute_priority, kvx_partition **out, char *msg,
                                size_t msg_len)
{
    if (msg && msg_len)
        msg[0] = '\0';
    if (!out || io_sms <= 0 || io_groups <= 0 || io_groups > kvx_partition::kMaxGroups)
        return KVX_ERR_INVALID_ARG;
    *out = nullptr;
    Driver d;
    if (!load_driver(&d))
        return fail(msg, msg_len, "green-context driver entry points unavailable");
    int prev = -1;
    cudaGetDevice(&prev);
    if (cudaSetDevice(device) != cudaSuccess || cudaFree(nullptr) != cudaSuccess) {
        cudaGetLastError();
        return fail(msg, msg_len, "cannot initialise device %d", device);
    }
    kvx_partition *p = new kvx_partition();
    p->device = device;
    p->groups = io_groups;
    CUdevice dev;
    CUdevResource all, io[kvx_partition::kMaxGroups], rest;
    std::memset(&all, 0, sizeof all);
    std::memset(io, 0, sizeof io);
    std::memset(&rest, 0, sizeof rest);
    unsigned int groups = unsigned(io_groups);
    const char *step = "cuDeviceGet";
    CUresult r = d.device_get(&dev, device);
    if (r == CUDA_SUCCESS) {
        step = "cuDeviceGetDevResource";
        r = d.get_dev_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM);
    }
    if (r == CUDA_SUCCESS) {
        step = "cuDevSmResourceSplitByCount";
        r = d.split_by_count(io, &groups, &all, &rest, 0, unsigned(io_sms));
    }
    if (r == CUDA_SUCCESS && (groups != unsigned(io_groups) || rest.sm.smCount == 0)) {
        delete p;
        if (prev >= 0)
            cudaSetDevice(prev);
        return fail(msg, msg_len, "cannot split %u SMs into %d groups of %d I/O SMs and a "
                    "remainder", all.sm.smCount, io_groups, io_sms);
    }
    for (int g = 0; g <= io_groups && r == CUDA_SUCCESS; ++g) {
        CUdevResource *res = g < io_groups ? &io[g] : &rest;
        CUdevResourceDesc desc = nullptr;
        step = "cuDevResourceGenerateDesc";
        r = d.generate_desc(&desc, res, 1);
        if (r == CUDA_SUCCESS) {
            step = "cuGreenCtxCreate";
            r = d.green_create(&p->ctx[g], desc, dev, CU_GREEN_CTX_DEFAULT_STREAM);
        }
        if (r == CUDA_SUCCESS) {
            step = "cuGreenCtxStreamCreate";
            r = d.green_stream_create(&p->stream[g], p->ctx[g], CU_STREAM_NON_BLOCKING,
                                      g < io_groups ? io_priority : compute_priority);
        }
        p->sms[g] = int(res->sm.smCount);
    }
    if (prev >= 0)
        cudaSetDevice(prev);
    if (r != CUDA_SUCCESS) {
        release(d, p);
        delete p;
        return fail(msg, msg_len, "%s failed with CUresult %d", step, int(r));
    }
    *out = p;
    return KVX_OK;
}

kvx_status kvx_partition_info(const kvx_partition *p, int group, kvx_stream_t *stream,
                              int *sms)
{
    if (!p || group < 0 || group > p->groups)
        return KVX_ERR_INVALID_ARG;
    if (stream)
        *stream = reinterpret_cast<kvx_stream_t>(p->stream[group]);
    if (sms)
        *sms = p->sms[group];
    return KVX_OK;
}

void kvx_partition_destroy(kvx_partition *p)
{
    if (!p)
        return;
    Driver d;
    if (load_driver(&d)) {
        int prev = -1;
        cudaGetDevice(&prev);
        cudaSetDevice(p->device);
        cudaDeviceSynchronize();
        release(d, p);
        if (prev >= 0)
            cudaSetDevice(prev);
    }
    delete p;
}

}  // extern "C"
