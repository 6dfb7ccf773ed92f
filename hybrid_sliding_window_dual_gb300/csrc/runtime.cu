// Runtime plumbing of libhswa: device error word, tensor-map encoding,
// dispatch trace, and the upload of the pool's block tables.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace hswa {

// One error word per device (module globals are per device).
__device__ int g_error_word = 0;

namespace {
int *g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mu;
thread_local const char *g_last_kernel = "";
thread_local const char *g_last_cuda_error = "";
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}
std::mutex g_setup_mu;
}  // namespace

int device_index() { return current_device(); }

std::mutex &setup_mutex() { return g_setup_mu; }

int *error_word() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int *>(p);
    }
    return g_err_ptr[dev];
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

void set_last_kernel(const char *name) { g_last_kernel = name; }

int cuda_fail(cudaError_t e, const char *where) {
    static thread_local char buf[256];
    snprintf(buf, sizeof(buf), "%s: %s", where, cudaGetErrorString(e));
    g_last_cuda_error = buf;
    return HSWA_ERR_CUDA;
}

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

static size_t elem_bytes(CUtensorMapDataType t) {
    return t == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : t == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2;
}

bool make_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols, CUtensorMapDataType type, CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem_bytes(type)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                  uint32_t b1, uint32_t b2, CUtensorMapDataType type, CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc) return false;
    const uint64_t es = elem_bytes(type);
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, type, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Apply a list of (flat index, value) updates to the three device arrays
// [full_bt | swa_bt | seq_len]. Each index appears at most once.
__global__ void apply_table_updates(const int64_t *__restrict__ idx, const int32_t *__restrict__ val, int64_t n,
                                    int64_t table_entries, int32_t *full_bt, int32_t *swa_bt, int32_t *seq_len) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t f = idx[i];
        if (f < table_entries)
            full_bt[f] = val[i];
        else if (f < 2 * table_entries)
            swa_bt[f - table_entries] = val[i];
        else
            seq_len[f - 2 * table_entries] = val[i];
    }
}

// Waits on an mbarrier that nothing completes, with the same bounded wait
// the attention kernels use: it must give up, record HSWA_ERR_TIMEOUT and
// return, leaving the context usable.
__global__ void selftest_bounded_wait(int *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err);
}

}  // namespace hswa

using namespace hswa;

extern "C" int hswa_selftest_bounded_wait(hswa_stream_t stream) {
    HSWA_NVTX("hswa_selftest_bounded_wait");
    int *err = error_word();
    if (!err) return HSWA_ERR_CUDA;
    set_last_kernel("selftest_bounded_wait");
    selftest_bounded_wait<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? HSWA_OK : HSWA_ERR_CUDA;
}

void hswa_pool_release_device(hswa_pool *pool) {
    if (pool->staging_event) {
        cudaEventSynchronize(static_cast<cudaEvent_t>(pool->staging_event));
        cudaEventDestroy(static_cast<cudaEvent_t>(pool->staging_event));
        pool->staging_event = nullptr;
    }
    if (pool->staging) {
        cudaFreeHost(pool->staging);
        pool->staging = nullptr;
    }
}

extern "C" int hswa_sync_tables(hswa_pool *pool, int32_t *d_full_bt, int32_t *d_swa_bt, int32_t *d_seq_len,
                                hswa_stream_t stream) {
    HSWA_NVTX("hswa_sync_tables");
    if (!pool || !d_full_bt || !d_swa_bt || !d_seq_len) return HSWA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t E = pool->table_entries();
    if (d_full_bt != pool->last_dev[0] || d_swa_bt != pool->last_dev[1] || d_seq_len != pool->last_dev[2])
        pool->need_full_upload = true;
    set_last_kernel("sync_tables");
    if (pool->need_full_upload) {
        // whole tables, straight from the host mirrors (synchronous copies)
        if (cudaMemcpyAsync(d_full_bt, pool->full_bt.data(), E * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(d_swa_bt, pool->swa_bt.data(), E * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(d_seq_len, pool->seq_len.data(), pool->cfg.max_seqs * 4, cudaMemcpyHostToDevice,
                            st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return HSWA_ERR_CUDA;
        for (int64_t f : pool->dirty_list) pool->dirty_flag[f] = 0;
        pool->dirty_list.clear();
        pool->last_dev[0] = d_full_bt;
        pool->last_dev[1] = d_swa_bt;
        pool->last_dev[2] = d_seq_len;
        pool->need_full_upload = false;
        return HSWA_OK;
    }
    const int64_t n = (int64_t)pool->dirty_list.size();
    if (n == 0) return HSWA_OK;
    const size_t need = (size_t)n * (sizeof(int64_t) + sizeof(int32_t)) + 16;
    if (pool->staging_event &&
        cudaEventSynchronize(static_cast<cudaEvent_t>(pool->staging_event)) != cudaSuccess)
        return HSWA_ERR_CUDA;
    if (need > pool->staging_bytes) {
        if (pool->staging) cudaFreeHost(pool->staging);
        pool->staging = nullptr;
        const size_t cap = std::max(need * 2, (size_t)1 << 16);
        if (cudaHostAlloc(&pool->staging, cap, cudaHostAllocDefault) != cudaSuccess) {
            pool->staging_bytes = 0;
            return HSWA_ERR_CUDA;
        }
        pool->staging_bytes = cap;
    }
    if (!pool->staging_event) {
        cudaEvent_t ev;
        if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return HSWA_ERR_CUDA;
        pool->staging_event = ev;
    }
    int64_t *h_idx = static_cast<int64_t *>(pool->staging);
    int32_t *h_val = reinterpret_cast<int32_t *>(h_idx + n);
    for (int64_t i = 0; i < n; ++i) {
        const int64_t f = pool->dirty_list[i];
        h_idx[i] = f;
        h_val[i] = f < E ? pool->full_bt[f] : f < 2 * E ? pool->swa_bt[f - E] : pool->seq_len[f - 2 * E];
        pool->dirty_flag[f] = 0;
    }
    pool->dirty_list.clear();
    // the kernel reads the packed updates straight from the pinned buffer
    // through its device-mapped address
    int64_t *d_idx = nullptr;
    if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&d_idx), pool->staging, 0) != cudaSuccess)
        return HSWA_ERR_CUDA;
    const int32_t *d_val = reinterpret_cast<const int32_t *>(d_idx + n);
    const int threads = 256;
    const int blocks = (int)std::min<int64_t>((n + threads - 1) / threads, 1024);
    apply_table_updates<<<blocks, threads, 0, st>>>(d_idx, d_val, n, E, d_full_bt, d_swa_bt, d_seq_len);
    if (cudaGetLastError() != cudaSuccess) return HSWA_ERR_CUDA;
    if (cudaEventRecord(static_cast<cudaEvent_t>(pool->staging_event), st) != cudaSuccess) return HSWA_ERR_CUDA;
    return HSWA_OK;
}

extern "C" int hswa_check(hswa_stream_t stream) {
    HSWA_NVTX("hswa_check");
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return HSWA_ERR_CUDA;
    int *w = error_word();
    if (!w) return HSWA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return HSWA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return HSWA_ERR_CUDA;
    }
    return v;
}

extern "C" const char *hswa_last_kernel(void) { return g_last_kernel; }

extern "C" const char *hswa_last_cuda_error(void) { return g_last_cuda_error; }
