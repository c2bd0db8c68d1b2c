// api.cu -- status strings, device status read-back, the wait bound, and the grid-wait self test.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

#include "host_util.h"

namespace dspark {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<uint64_t> g_launches{0};
int g_sm_count[64] = {0};

__global__ void selftest_grid_wait_kernel(WsHeader* hdr, uint32_t expected, uint64_t limit_ns, int32_t* passed) {
    if (grid_wait(hdr, expected, limit_ns) && threadIdx.x == 0) atomicAdd(passed, 1);
}
}  // namespace

cudaError_t device_sm_count(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && g_sm_count[dev] > 0) {
        *sms = g_sm_count[dev];
        return cudaSuccess;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_sm_count[dev] = n;
    *sms = n;
    return cudaSuccess;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }


namespace {
struct KernelPrep {
    int dev;
    const void* fn;
    size_t smem_set;  // largest dynamic shared memory granted so far
    size_t smem;
    int threads;
    int per_sm;
};
std::mutex g_prep_mu;
std::vector<KernelPrep> g_prep;
}  // namespace

namespace {
struct ClusterOcc {
    int dev;
    const void* fn;
    int cs, threads;
    size_t smem;
    int n;
};
std::vector<ClusterOcc> g_cocc;
}  // namespace

cudaError_t max_active_clusters(const void* fn, int cs, int threads, size_t smem, int* n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_prep_mu);
    for (const ClusterOcc& c : g_cocc)
        if (c.dev == dev && c.fn == fn && c.cs == cs && c.threads == threads && c.smem == smem) {
            *n = c.n;
            return cudaSuccess;
        }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int k = 0;
    if (cudaOccupancyMaxActiveClusters(&k, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();  // an unsupported shape: remember it as zero
        k = 0;
    }
    g_cocc.push_back(ClusterOcc{dev, fn, cs, threads, smem, k});
    *n = k;
    return cudaSuccess;
}

cudaError_t prepare_kernel(const void* fn, size_t smem, int threads, int* per_sm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_prep_mu);
    size_t granted = 0;
    for (const KernelPrep& k : g_prep)
        if (k.dev == dev && k.fn == fn) {
            if (k.smem == smem && k.threads == threads) {
                *per_sm = k.per_sm;
                return cudaSuccess;
            }
            granted = granted > k.smem_set ? granted : k.smem_set;
        }
    if (smem > granted) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        granted = smem;
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
    if (e != cudaSuccess) return e;
    g_prep.push_back(KernelPrep{dev, fn, granted, smem, threads, n});
    *per_sm = n;
    return cudaSuccess;
}

}  // namespace dspark

using namespace dspark;

extern "C" void dspark_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

extern "C" dspark_status dspark_get_device_status(const void* workspace, dspark_stream_t stream, int32_t* out) {
    if (!workspace || !out) return DSPARK_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
    *out = v;
    return DSPARK_OK;
}

extern "C" dspark_status dspark_selftest_grid_wait(int nblocks, int missing, void* workspace, size_t ws_bytes,
                                                   dspark_stream_t stream) {
    if (nblocks < 1 || missing < 0) return DSPARK_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < kHeaderBytes + 256) return DSPARK_ERR_WORKSPACE;
    int sms = 0;
    if (device_sm_count(&sms) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (nblocks > sms) return DSPARK_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes + 256, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    WsHeader* hdr = static_cast<WsHeader*>(workspace);
    uint32_t expected = (uint32_t)(nblocks + missing);
    uint64_t limit = wait_limit_ns();
    int32_t* passed = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + kHeaderBytes);
    void* args[] = {&hdr, &expected, &limit, &passed};
    if (cudaLaunchCooperativeKernel((const void*)selftest_grid_wait_kernel, dim3(nblocks), dim3(64), args, 0, s) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}

extern "C" uint64_t dspark_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char* dspark_status_string(dspark_status s) {
    switch (s) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID_ARG: return "invalid argument";
        case DSPARK_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case DSPARK_ERR_CUDA: return "CUDA runtime error";
        case DSPARK_ERR_TIMEOUT: return "device wait timed out";
        case DSPARK_ERR_BUDGET: return "verify budget smaller than the number of requests";
        case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DSPARK_ERR_TOKEN_RANGE: return "token id out of range or too few target rows";
        default: return "unknown status";
    }
}
