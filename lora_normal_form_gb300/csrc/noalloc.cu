// Token indexing without a context and without any device allocation.
//
// Who calls this: a batch scheduler or router that shares the GPU with a
// serving engine that has already reserved its memory pool (most of HBM for
// the KV cache), so a fresh allocation would fail or eat memory the pool
// relies on; and latency-critical code, where cudaMalloc/cudaFree may
// synchronise the device.  A context cannot serve them: creating one allocates
// its workspaces.  The indexing kernel itself only needs two small pieces of
// device scratch besides the caller's outputs, the adapter -> method table and
// a status word, so they live in one file-scope device array per device.
#include <mutex>

#include <cuda_runtime.h>

#include "scute.h"
#include "internal.h"

namespace scute {
namespace {

constexpr int MAX_DEVICES = 64;
constexpr size_t TABLE_OFFSET = 256;   // status word in the first 256 bytes
static_assert(SCUTE_NOALLOC_SCRATCH_BYTES == TABLE_OFFSET + SCUTE_NOALLOC_MAX_ADAPTERS,
              "scratch layout: status block, then one int8 per adapter id");
static_assert(SCUTE_NOALLOC_MAX_ADAPTERS * (N_RANKS) < 65536,
              "the sort packs (method, id) into 16 bits");
static_assert((int)SCUTE_LORA == (int)RANK_LORA && (int)SCUTE_DORA == (int)RANK_DORA && (int)SCUTE_IA3 == (int)RANK_IA3 &&
                  (int)SCUTE_VERA == (int)RANK_VERA && (int)SCUTE_OFT == (int)RANK_OFT && (int)SCUTE_NF == (int)RANK_NF,
              "method codes are the kernel's method ranks");

// [0, 4): status word (must start at zero: the kernel only ORs bits into it);
// [256, 256 + n_adapters): method rank of each adapter id (-1: none).
__device__ __align__(256) unsigned char g_noalloc_scratch[SCUTE_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_addr[MAX_DEVICES];   // device address of the array, per device

}  // namespace
}  // namespace scute

using namespace scute;

extern "C" scute_status scute_index_tokens_noalloc(const int8_t *method_of_adapter, int32_t n_adapters,
                                                   const int32_t *adapter_ids, int64_t n, int32_t *perm,
                                                   int32_t *aid_sorted, int32_t *seg_start, int32_t *seg_aid,
                                                   int32_t *counts, int32_t *flags, void *stream) {
    if (n < 0 || n_adapters < 1 || !method_of_adapter || !seg_start || !counts ||
        (n > 0 && (!adapter_ids || !perm || !aid_sorted || !seg_aid)))
        return SCUTE_ERR_ARG;
    if (n > SCUTE_MAX_TOKENS || n_adapters > SCUTE_NOALLOC_MAX_ADAPTERS) return SCUTE_ERR_UNSUPPORTED;
    for (int32_t a = 0; a < n_adapters; ++a)
        if (method_of_adapter[a] < -1 || method_of_adapter[a] > SCUTE_NF) return SCUTE_ERR_ARG;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SCUTE_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= MAX_DEVICES) return SCUTE_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return SCUTE_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return SCUTE_ERR_NO_DEVICE;

    unsigned char *base;
    {
        // one lookup per device, made with that device current (it is: dev is
        // the current device); later calls reuse the address
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_addr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return SCUTE_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
        }
        base = static_cast<unsigned char *>(g_scratch_addr[dev]);
    }
    int *status = reinterpret_cast<int *>(base);
    int8_t *table = reinterpret_cast<int8_t *>(base + TABLE_OFFSET);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // scute_method codes equal the kernel's method ranks (LoRA 0 ... NF 5), so
    // the caller's table is used as it is
    cudaGetLastError();
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess ||
        cudaMemcpyAsync(table, method_of_adapter, (size_t)n_adapters, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        launch_index(adapter_ids, (int)n, table, n_adapters, perm, aid_sorted, seg_start, seg_aid,
                     reinterpret_cast<IndexMeta *>(counts), status, st) != cudaSuccess ||
        (flags && cudaMemcpyAsync(flags, status, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)) {
        cudaGetLastError();
        return SCUTE_ERR_CUDA;
    }
    return SCUTE_OK;
}
