// Sparse decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a CUDA
// graph being captured, an engine whose memory planner owns every byte of the
// device and forbids outside allocations, or a process that has handed all free
// memory to a pooling allocator.  ckv_sparse_decode_attn needs a context, and
// creating one allocates the split-K workspace.  This entry point runs the same
// attention kernel without a context: its only scratch (the per-split partial
// results that the combine kernel merges) lives in one fixed-size array in the
// library's own device memory, reserved when the library is loaded and kept
// until the process exits.  The array's address is looked up once per device
// in the device's primary context (the one the runtime API uses); a
// cudaDeviceReset invalidates it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t SCRATCH_BYTES = (size_t)8 << 20;  // 8 MiB per device that loads the library
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[SCRATCH_BYTES];

std::mutex g_lock;
void* g_scratch_addr[MAX_DEVICES];
int g_num_sms[MAX_DEVICES];

// Device address of the scratch array on the current device (and the device's
// SM count), looked up once per device: the host-side symbol is only a
// stand-in, never a device address.
cudaError_t scratch_address(void** out, int* num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_num_sms[dev] = sms;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    *num_sms = g_num_sms[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ckv_status ckv_sparse_decode_attn_noalloc(const void* q, int32_t q_dtype, const void* K,
                                                     const void* V, const int32_t* idx,
                                                     const int32_t* count, int32_t units, int32_t g,
                                                     int32_t max_len, int32_t sinks, int32_t clustered_end,
                                                     int32_t cur_len, int32_t B, float* out,
                                                     int32_t* dev_err, void* stream) {
    CKV_TRACE("ckv_sparse_decode_attn_noalloc");
    using namespace ckv;
    if (!q || !K || !V || !idx || !count || !out) return CKV_ERR_ARG;
    if (q_dtype != CKV_F32 && q_dtype != CKV_BF16) return CKV_ERR_DTYPE;
    if (g != 1 && g != 2 && g != 4 && g != 8) return CKV_ERR_ARG;
    if (units < 1 || sinks < 0 || B < 0 || clustered_end < sinks || cur_len < clustered_end ||
        cur_len > max_len)
        return CKV_ERR_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return CKV_ERR_ALIGN;

    const int rs = attention_rows_per_split(q_dtype, g);
    const long long rows = (long long)sinks + (cur_len - clustered_end) + B;
    const long long splits = (rows + rs - 1) / rs;
    const long long need = (long long)units * splits * g * (D + 2) * (long long)sizeof(float);
    if (need > (long long)SCRATCH_BYTES) return CKV_ERR_CAPACITY;

    void* base = nullptr;
    int num_sms = 0;
    if (scratch_address(&base, &num_sms) != cudaSuccess) return CKV_ERR_CUDA;
    // every partial the combine reads is written by the same call first: what
    // the previous call left in the array is never read
    float* part = static_cast<float*>(base);
    cudaStream_t s = (cudaStream_t)stream;
    const cudaError_t e = launch_attention(q, K, V, idx, count, units, g, q_dtype, max_len, sinks, clustered_end,
                                           cur_len, B, out, part, (int)splits, dev_err, num_sms, WAIT_LIMIT, 0, s);
    return e == cudaSuccess ? CKV_OK : CKV_ERR_CUDA;
}
