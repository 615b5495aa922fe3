// qdec_static_scratch.cu -- qdec_step for callers that cannot allocate
// device memory.
//
// qdec_step needs a scratch workspace (per-piece partial results and one
// arrival counter per (sequence, KV head)), which its caller normally
// allocates.  Some callers have no allocator to give: code that runs while
// the process is already inside a latency-critical serving loop where
// cudaMalloc/cudaFree would synchronise the device, plugins hosted by a
// runtime that owns every device allocation and exposes none to them, or
// embeddings that size all device memory once at start-up.  For them the
// scratch lives in a fixed array in this library's own device memory,
// reserved when the library is loaded and held until the process exits.
//
// This entry point allocates nothing: it reuses qdec_step's kernel and
// launch path unchanged and only supplies the array as the workspace.
#include "qdec_internal.h"
#include "qdec.h"

#include <mutex>

namespace {

// The scratch itself.  Host code must not use this name as a pointer (on
// the host it is only a stand-in for the symbol); its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[QDEC_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_addr[64];  // device address of the array, per device id

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached.
qdec_status scratch_address(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QDEC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        // An error the caller has not read yet stays pending; only the one
        // this lookup raised is cleared.
        const cudaError_t pending = cudaPeekAtLastError();
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            if (pending == cudaSuccess) cudaGetLastError();
            return QDEC_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *addr = g_scratch_addr[dev];
    return QDEC_OK;
}

}  // namespace

extern "C" qdec_status qdec_step_static_scratch(
    const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride, const qdec_bf16 *k,
    int64_t k_stride, const qdec_bf16 *v, int64_t v_stride, const qdec_bf16 *q_norm_w,
    const qdec_bf16 *k_norm_w, const int32_t *positions, const int32_t *seq_lens,
    const int32_t *block_table, const void *rope_table, qdec_bf16 *kv_pool, qdec_bf16 *out,
    int32_t *err_flag, void *stream) {
    const size_t need = qdec_workspace_bytes(shape);
    if (need == 0)  // invalid shape: let qdec_step name the problem
        return qdec_step(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w,
                         positions, seq_lens, block_table, rope_table, kv_pool, nullptr, 0, out,
                         err_flag, stream);
    if (need > static_cast<size_t>(QDEC_STATIC_SCRATCH_BYTES)) return QDEC_ERR_WORKSPACE;
    void *ws = nullptr;
    const qdec_status st = scratch_address(&ws);
    if (st != QDEC_OK) return st;
    // The array keeps whatever the previous call left; the arrival counters
    // at its front must start at zero.
    const qdec_status cleared = qdec_workspace_init(shape, ws, need, stream);
    if (cleared != QDEC_OK) return cleared;
    return qdec_step(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w, positions,
                     seq_lens, block_table, rope_table, kv_pool, ws, need, out, err_flag, stream);
}
