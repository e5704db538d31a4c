// paged_decode_attention_static: decode attention whose scratch memory (the work
// counters and the split-context partials) lives in a fixed, file-scope device array,
// so neither the caller nor the library allocates anything during the call.
//
// For callers that cannot call cudaMalloc: plugins or embedded components whose host
// application owns all device memory and hands them no allocator, and serving loops
// that forbid device allocation once they are running (cudaMalloc can synchronise the
// device, stall on fragmentation, or fail late).  Such a caller still passes its own
// inputs and outputs; only the scratch comes from here.
//
// The array is KV_STATIC_SCRATCH_BYTES long.  Every GPU that loads this library holds
// it until the process exits.  All calls share it: a call's partials stay in it after
// the call, the work counters are cleared at the start of every call, and two calls
// whose kernels overlap on the GPU (different streams, or different host threads)
// race on it.

#include <mutex>

#include "kvp_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char kv_static_scratch[KV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // context the address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the current context, 0 if it cannot be read.  A context created
// after cudaDeviceReset gets a new id, so an address looked up in the old one is never
// reused.  The two driver entry points are fetched on the first call (with g_scratch_mu held).
unsigned long long current_context_id() {
    static bool tried = false;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!tried) {
        tried = true;
        void* f0 = nullptr;
        void* f1 = nullptr;
        cudaDriverEntryPointQueryResult q0, q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &q0) == cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            q0 == cudaDriverEntryPointSuccess && q1 == cudaDriverEntryPointSuccess && f0 && f1) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(f0);
            get_id = reinterpret_cast<CtxGetIdFn>(f1);
        } else {
            cudaGetLastError();
        }
    }
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on the current device `dev`.  In host code the
// name kv_static_scratch is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, with that device current.  It is looked up once per device and
// context: on the first call on a device, and again on the first call after the device's
// context was replaced (cudaDeviceReset), or on every call if the context id cannot be read.
int scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return KV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, kv_static_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            g_scratch_ptr[dev] = nullptr;
            return KV_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return KV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_static(kv_pool* pool, int layer, const void* q, float* out,
                                             const int32_t* block_tables, int max_blocks_per_seq,
                                             const int32_t* context_lens, int batch, int max_context,
                                             float scale, int partition_tokens, kv_stream_t stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers || batch < 0 || max_context < 0)
        return KV_ERR_INVALID_ARG;
    if (batch == 0) return KV_OK;
    if (!q || !out || !block_tables || !context_lens || max_blocks_per_seq < 1) return KV_ERR_INVALID_ARG;
    if (!kvp::aligned16(q) || !kvp::aligned16(out)) return KV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return KV_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
    if (dev != pool->device) return KV_ERR_INVALID_ARG;      // the pool's device must be current
    kvp::AttnPlan plan;
    int rc = kvp::plan_attention(pool, batch, max_context, partition_tokens, &plan);
    if (rc != KV_OK) return rc;
    if (plan.ws_bytes > KV_STATIC_SCRATCH_BYTES) return KV_ERR_INVALID_ARG;   // does not fit
    void* scratch = nullptr;
    rc = scratch_address(dev, &scratch);
    if (rc != KV_OK) return rc;
    return kvp::launch_attention(pool, layer, q, out, block_tables, max_blocks_per_seq, context_lens,
                                 batch, max_context, scale, plan, scratch, stream);
}
