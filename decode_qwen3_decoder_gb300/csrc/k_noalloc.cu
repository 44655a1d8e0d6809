// LM head + greedy argmax for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need a result: a plugin that
// runs inside another framework's memory manager with a fixed device budget, a serving loop
// that must never touch the allocator after start-up (an allocation can synchronise the
// device and stall every stream), or code that prepares work while a stream is being
// captured. For them this file offers a variant of the small-batch LM-head kernel whose
// only scratch, the packed per-row argmax keys, lives in a file-scope __device__ array
// instead of the model workspace. The caller still passes the input rows and the outputs.
//
// The array is QW_NOALLOC_MAX_ROWS 64-bit keys; every GPU that loads the library holds it
// until the process exits. All calls share it and it keeps the last call's contents, so
// each call clears the keys it uses before the kernel runs (and the unpack kernel zeroes
// them again afterwards). Calls whose work overlaps on the GPU race on the array.
#include <mutex>

#include "qw_internal.h"

static __device__ __align__(256) unsigned long long g_noalloc_keys[QW_NOALLOC_MAX_ROWS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_keys_addr[kMaxDevices];  // device address of g_noalloc_keys, per device

// Turn the packed keys into ids (lowest index wins ties) and clear them.
__global__ void k_noalloc_unpack(unsigned long long* keys, int B, int32_t* next_ids) {
    const int b = threadIdx.x;
    if (b < B) {
        const unsigned long long key = keys[b];
        next_ids[b] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
        keys[b] = 0ull;
    }
}

}  // namespace

extern "C" qw_status qw_lm_head_argmax_noalloc(const qw_model* m, int B, const float* dev_x, float* dev_logits,
                                               int32_t* dev_next_ids, void* stream_) {
    LmHeadView v;
    if (!qw_model_lmhead_view(m, &v)) return qw_fail(QW_ERR_INVALID_ARG, "model is NULL");
    if (B < 1 || B > QW_NOALLOC_MAX_ROWS)
        return qw_fail(QW_ERR_INVALID_ARG, "B=%d outside [1, %d]: the static scratch holds %d rows", B,
                       QW_NOALLOC_MAX_ROWS, QW_NOALLOC_MAX_ROWS);
    if (!dev_x || !dev_next_ids) return qw_fail(QW_ERR_INVALID_ARG, "dev_x or dev_next_ids is NULL");
    if (((uintptr_t)dev_x & 15) || ((uintptr_t)dev_logits & 15))
        return qw_fail(QW_ERR_INVALID_ARG, "dev_x and dev_logits must be 16-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qw_fail(QW_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return qw_fail(QW_ERR_UNSUPPORTED, "device %d beyond the set-up table", dev);
    void* keys = nullptr;
    {
        // Once per device, with that device current: the host-side name of the array is
        // only a stand-in, so ask the runtime for its device address.
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_keys_addr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_keys);
            if (e != cudaSuccess || !p)
                return qw_fail(QW_ERR_CUDA, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            g_keys_addr[dev] = p;
        }
        keys = g_keys_addr[dev];
    }
    cudaStream_t st = (cudaStream_t)stream_;
    e = cudaMemsetAsync(keys, 0, (size_t)B * sizeof(unsigned long long), st);
    if (e != cudaSuccess) return qw_fail(QW_ERR_CUDA, "clearing the keys failed: %s", cudaGetErrorString(e));
    LaunchCtx c = {st, false, nullptr};
    e = launch_gemv_lmhead(c, B, dev_x, nullptr, v.final_norm, v.eps, v.embed, v.vocab, v.hidden, dev_logits,
                           (unsigned long long*)keys);
    if (e != cudaSuccess) return qw_fail(QW_ERR_CUDA, "LM-head launch failed: %s", cudaGetErrorString(e));
    k_noalloc_unpack<<<1, 32, 0, st>>>((unsigned long long*)keys, B, dev_next_ids);
    e = cudaGetLastError();
    if (e != cudaSuccess) return qw_fail(QW_ERR_CUDA, "unpack launch failed: %s", cudaGetErrorString(e));
    return QW_OK;
}
