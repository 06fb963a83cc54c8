// kvx_partition.cpp -- hard SM partitioning for I/O vs compute with green contexts.
//
// "Tutti: Making SSD-Backed KV Cache Practical for Long-Context LLM Serving", section 2
// Design 2, splits the GPU's SMs into a compute domain and an I/O domain with NVIDIA green
// contexts so that the I/O kernel never competes with compute for SMs.  Here the device's
// SM resource is split into an I/O partition of at least `io_sms` SMs (the driver rounds
// up to its partition granularity) and a compute partition with the rest; each becomes a
// green context with one non-blocking stream.  Transfers launched on the I/O stream run
// only on the I/O SMs; anything launched on the compute stream (a GEMM, attention) runs
// only on the others.
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
    int device = 0;
    CUgreenCtx io_ctx = nullptr;
    CUgreenCtx compute_ctx = nullptr;
    CUstream io_stream = nullptr;
    CUstream compute_stream = nullptr;
    int io_sms = 0;
    int compute_sms = 0;
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
    if (p->io_stream)
        d.stream_destroy(p->io_stream);
    if (p->compute_stream)
        d.stream_destroy(p->compute_stream);
    if (p->io_ctx)
        d.green_destroy(p->io_ctx);
    if (p->compute_ctx)
        d.green_destroy(p->compute_ctx);
}

}  // namespace

extern "C" {

kvx_status kvx_partition_create(int device, int io_sms, int io_priority, int compute_priority,
                                kvx_partition **out, char *msg, size_t msg_len)
{
    if (msg && msg_len)
        msg[0] = '\0';
    if (!out || io_sms <= 0)
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
    CUdevice dev;
    CUdevResource all, io, rest;
    std::memset(&all, 0, sizeof all);
    std::memset(&io, 0, sizeof io);
    std::memset(&rest, 0, sizeof rest);
    unsigned int groups = 1;
    CUdevResourceDesc io_desc = nullptr, rest_desc = nullptr;
    CUresult r = d.device_get(&dev, device);
    const char *step = "cuDeviceGet";
    if (r == CUDA_SUCCESS) {
        step = "cuDeviceGetDevResource";
        r = d.get_dev_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM);
    }
    if (r == CUDA_SUCCESS) {
        step = "cuDevSmResourceSplitByCount";
        r = d.split_by_count(&io, &groups, &all, &rest, 0, unsigned(io_sms));
    }
    if (r == CUDA_SUCCESS && (groups != 1 || rest.sm.smCount == 0)) {
        release(d, p);
        delete p;
        if (prev >= 0)
            cudaSetDevice(prev);
        return fail(msg, msg_len, "cannot split %u SMs into %d I/O SMs and a remainder",
                    all.sm.smCount, io_sms);
    }
    if (r == CUDA_SUCCESS) {
        step = "cuDevResourceGenerateDesc";
        r = d.generate_desc(&io_desc, &io, 1);
        if (r == CUDA_SUCCESS)
            r = d.generate_desc(&rest_desc, &rest, 1);
    }
    if (r == CUDA_SUCCESS) {
        step = "cuGreenCtxCreate";
        r = d.green_create(&p->io_ctx, io_desc, dev, CU_GREEN_CTX_DEFAULT_STREAM);
        if (r == CUDA_SUCCESS)
            r = d.green_create(&p->compute_ctx, rest_desc, dev, CU_GREEN_CTX_DEFAULT_STREAM);
    }
    if (r == CUDA_SUCCESS) {
        step = "cuGreenCtxStreamCreate";
        r = d.green_stream_create(&p->io_stream, p->io_ctx, CU_STREAM_NON_BLOCKING, io_priority);
        if (r == CUDA_SUCCESS)
            r = d.green_stream_create(&p->compute_stream, p->compute_ctx, CU_STREAM_NON_BLOCKING,
                                      compute_priority);
    }
    if (prev >= 0)
        cudaSetDevice(prev);
    if (r != CUDA_SUCCESS) {
        release(d, p);
        delete p;
        return fail(msg, msg_len, "%s failed with CUresult %d", step, int(r));
    }
    p->io_sms = int(io.sm.smCount);
    p->compute_sms = int(rest.sm.smCount);
    *out = p;
    return KVX_OK;
}

kvx_status kvx_partition_info(const kvx_partition *p, kvx_stream_t *io_stream,
                              kvx_stream_t *compute_stream, int *io_sms, int *compute_sms)
{
    if (!p)
        return KVX_ERR_INVALID_ARG;
    if (io_stream)
        *io_stream = reinterpret_cast<kvx_stream_t>(p->io_stream);
    if (compute_stream)
        *compute_stream = reinterpret_cast<kvx_stream_t>(p->compute_stream);
    if (io_sms)
        *io_sms = p->io_sms;
    if (compute_sms)
        *compute_sms = p->compute_sms;
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
