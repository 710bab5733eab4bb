// dg_runtime.cu -- library-wide state: the device status word, device queries, tensor-map
// encoding, status strings and version.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "dg_common.cuh"

// One status word per device that loads the library; kernels receive its address.
static __device__ unsigned g_dg_status_word;

namespace {
constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_launches{0};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

namespace dghost {

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned* status_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dg_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_status_ptr[dev];
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

bool encode_tmap(void* tmap, int dtype_code, int rank, void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return false;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    CUtensorMapDataType dt = dtype_code == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
    else if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    else if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i > 0) gstride[i - 1] = strides_bytes[i - 1];
    }
    CUresult r = g_encode(static_cast<CUtensorMap*>(tmap), dt, (cuuint32_t)rank, base, gdim, gstride, bdim, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace dghost

namespace {
// The bounded waits of the kernels, run on shared-memory barriers of one warp: `never` gets
// no arrival (its waits must expire and raise DG_DEV_TIMEOUT, as in a kernel), `done` gets
// its one arrival before the wait (which must then succeed).
__global__ void k_probe_bounded_wait(unsigned* status, uint32_t polls, uint32_t* result) {
    __shared__ __align__(8) uint64_t never, done;
    if (threadIdx.x == 0) {
        dg::mbar_init(&never, 1);
        dg::mbar_init(&done, 1);
        dg::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) dg::mbar_arrive(&done);
    __syncwarp();
    uint32_t single = 1;
    if (threadIdx.x == 0) {
        single = dg::mbar_wait(&never, 0, polls) ? 1u : 0u;
        if (!single) dg::raise_status(status, DG_DEV_TIMEOUT);
    }
    const bool warp_ok = dg::mbar_wait_warp(&never, 0, 0, polls);
    const bool done_ok = dg::mbar_wait_warp(&done, 0, 0, polls);
    if (threadIdx.x == 0) {
        if (!warp_ok) dg::raise_status(status, DG_DEV_TIMEOUT);
        result[0] = single;
        result[1] = warp_ok ? 1u : 0u;
        result[2] = done_ok ? 1u : 0u;
    }
}
}  // namespace

extern "C" {

dg_status dg_probe_bounded_wait(uint32_t polls, uint32_t* result, dg_stream_t stream) {
    if (polls < 1 || polls > 65536 || !result) return DG_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(result) & 3u) return DG_ERR_ALIGNMENT;
    unsigned* st = dghost::status_word();
    if (!st) return DG_ERR_CUDA;
    k_probe_bounded_wait<<<1, 32, 0, (cudaStream_t)stream>>>(st, polls, result);
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

dg_status dg_get_device_status(dg_stream_t stream, uint32_t* status) {
    if (!status) return DG_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return DG_ERR_CUDA;
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_dg_status_word, sizeof v);
    if (e != cudaSuccess) return DG_ERR_CUDA;
    *status = v;
    return DG_OK;
}

dg_status dg_clear_device_status(dg_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return DG_ERR_CUDA;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_dg_status_word, &zero, sizeof zero);
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

const char* dg_status_string(dg_status s) {
    switch (s) {
        case DG_OK: return "DG_OK";
        case DG_ERR_INVALID_ARG: return "DG_ERR_INVALID_ARG";
        case DG_ERR_ALIGNMENT: return "DG_ERR_ALIGNMENT";
        case DG_ERR_WORKSPACE: return "DG_ERR_WORKSPACE";
        case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED";
        case DG_ERR_CUDA: return "DG_ERR_CUDA";
    }
    return "DG_UNKNOWN_STATUS";
}

int32_t dg_version(void) { return 100; }  // 0.1.0

uint64_t dg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
