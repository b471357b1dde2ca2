// ssd_noalloc.cu -- ssd_fwd_noalloc (include/ssd.h): the generic path with its
// scratch in a fixed device array that ships inside the library.
//
// Some callers may not allocate device memory themselves: a plug-in running
// inside a host application that owns the whole device-memory budget through
// its own pool, or a latency-bound loop in which cudaMalloc (which can
// synchronise the device) is not allowed.  This entry point needs no
// workspace from them.  It allocates nothing: the scratch is the array below,
// sized SSD_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library
// keeps until the process exits.  All calls share it, so calls that overlap on
// the GPU race; it keeps the previous call's contents, and the only part that
// must start at zero (the status word) is cleared by every call.
#include <cuda.h>

#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
// Per device: the array's device address and the unique ID of the context it was looked up in.
void *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}

// Unique ID of the calling thread's current context (0 when there is none or it cannot be read).
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_noalloc_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up with the device current.  It is cached
// together with the context it belongs to and looked up again when the current context differs
// (after cudaDeviceReset, or after the primary context was released and created anew, the
// module is loaded again and the array can move).
int scratch_on_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    const unsigned long long ctx = current_ctx_id();
    if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return SSD_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_ctx_id();   // the lookup makes the primary context current
    }
    *out = g_scratch_addr[dev];
    return SSD_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" int ssd_fwd_noalloc(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                               const void *B, const void *C, const float *D, const float *init_state,
                               void *y, float *final_state, void *stream) {
    Problem p;
    int st = validate_dims(dims, &p);
    if (st != SSD_OK) return st;
    if (dims->path == SSD_PATH_TCGEN05 || !generic_supports(p)) return SSD_ERR_UNSUPPORTED;
    const bool empty = (p.b == 0 || p.T == 0);
    if (!empty && (!x || !dt || !A || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    const void *ptrs[] = {x, dt, A, B, C, D, init_state, y, final_state};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return SSD_ERR_ALIGNMENT;
    if (!empty && y == x) return SSD_ERR_INVALID_ARG;
    if (generic_workspace_bytes(p) > SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_SCRATCH_LIMIT;

    void *ws = nullptr;
    if ((st = scratch_on_current_device(&ws)) != SSD_OK) return st;
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D;
    p.init = init_state; p.y = y; p.final_state = final_state;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (e != cudaSuccess) return note_cuda(e);
    e = empty ? launch_copy_state(p, s) : generic_launch(p, generic_carve(p, ws), s);
    return note_cuda(e);
}
