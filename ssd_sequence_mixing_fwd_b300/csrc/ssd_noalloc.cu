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
#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int scratch_on_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return SSD_ERR_CUDA;
        g_scratch_addr[dev] = p;
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
