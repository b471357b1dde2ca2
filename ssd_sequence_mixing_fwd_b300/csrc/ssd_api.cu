// ssd_api.cu -- the C ABI of libssd_b300 (declared in include/ssd.h):
// argument validation, workspace sizing, path selection and launches.
#include <atomic>
#include <cstring>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

std::atomic<int64_t> g_spin_limit{0};
std::atomic<int64_t> g_withhold{-1};
std::atomic<uint64_t> g_launches{0};
std::atomic<void *> g_ev_start{nullptr};
std::atomic<void *> g_ev_stop{nullptr};
std::atomic<int> g_last_cuda{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side checks of ssd_dims; fills *prob (pointers left null).
int check_dims(const ssd_dims *d, Problem *prob) {
    if (!d) return SSD_ERR_INVALID_ARG;
    if (d->b < 0 || d->T < 0 || d->H < 1 || d->G < 1 || d->P < 1 || d->N < 1) return SSD_ERR_INVALID_ARG;
    if (d->H % d->G != 0) return SSD_ERR_INVALID_ARG;
    if (d->Q != 64 && d->Q != 128 && d->Q != 256) return SSD_ERR_INVALID_ARG;
    if (d->a_mode != SSD_A_SCALAR && d->a_mode != SSD_A_DIAGONAL) return SSD_ERR_INVALID_ARG;
    if (d->io_dtype != SSD_DTYPE_BF16 && d->io_dtype != SSD_DTYPE_F32) return SSD_ERR_INVALID_ARG;
    if (d->path != SSD_PATH_AUTO && d->path != SSD_PATH_GENERIC && d->path != SSD_PATH_TCGEN05)
        return SSD_ERR_INVALID_ARG;
    if (d->reserved != 0) return SSD_ERR_INVALID_ARG;
    // Sizes whose element counts would overflow int64 indexing are rejected.
    const double elems = (double)d->b * (double)d->T * (double)d->H * (double)d->P;
    if (elems > 9.0e15 || (double)d->b * d->T * d->G * d->N > 9.0e15) return SSD_ERR_INVALID_ARG;
    std::memset(prob, 0, sizeof(*prob));
    prob->b = d->b; prob->T = d->T; prob->H = d->H; prob->P = d->P;
    prob->N = d->N; prob->G = d->G; prob->Q = d->Q;
    prob->nc = (d->T + d->Q - 1) / d->Q;
    prob->a_mode = d->a_mode;
    prob->io_dtype = d->io_dtype;
    if (d->P > 256 || (d->P & (d->P - 1)) || d->N > 256 || d->N * d->P > 16384) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// Which path runs for these dims (after check_dims succeeded).
int choose_path(const ssd_dims *d, const Problem &p, int32_t *path) {
    const bool tc = fused_supports(p) || diag_supports(p);
    const bool gen = generic_supports(p);
    if (d->path == SSD_PATH_TCGEN05) {
        if (!tc) return SSD_ERR_UNSUPPORTED;
        *path = SSD_PATH_TCGEN05;
    } else if (d->path == SSD_PATH_GENERIC) {
        if (!gen) return SSD_ERR_UNSUPPORTED;
        *path = SSD_PATH_GENERIC;
    } else {
        if (tc) *path = SSD_PATH_TCGEN05;
        else if (gen) *path = SSD_PATH_GENERIC;
        else return SSD_ERR_UNSUPPORTED;
    }
    return SSD_OK;
}

size_t workspace_for(const Problem &p, int32_t path) {
    if (path == SSD_PATH_TCGEN05) return diag_supports(p) ? diag_workspace_bytes(p) : fused_workspace_bytes(p);
    return generic_workspace_bytes(p);
}

__global__ void copy_state_kernel(const float *init, float *out, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = init ? init[i] : 0.f;
}

}  // namespace

cudaError_t launch_copy_state(const Problem &p, cudaStream_t s) {
    const int64_t n = p.b * p.H * p.N * p.P;
    if (!p.final_state || n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    copy_state_kernel<<<(unsigned)blocks, 256, 0, s>>>(p.init, p.final_state, n);
    note_launches(1);
    return cudaGetLastError();
}

void note_launches(int n) { g_launches.fetch_add((uint64_t)n); }
int note_cuda(cudaError_t e) {
    if (e != cudaSuccess) g_last_cuda.store((int)e);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
void record_dominant_start(cudaStream_t s) {
    void *a = g_ev_start.load(), *b = g_ev_stop.load();
    if (a && b) cudaEventRecord(static_cast<cudaEvent_t>(a), s);
}
void record_dominant_stop(cudaStream_t s) {
    void *a = g_ev_start.load(), *b = g_ev_stop.load();
    if (a && b) cudaEventRecord(static_cast<cudaEvent_t>(b), s);
}

int validate_dims(const ssd_dims *d, Problem *prob) { return check_dims(d, prob); }

int64_t debug_spin_limit() { return g_spin_limit.load(); }
int64_t debug_withhold_chunk() { return g_withhold.load(); }

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_abi_version(void) { return SSD_ABI_VERSION; }

extern "C" const char *ssd_status_string(int status) {
    switch (status) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported dimensions or path";
        case SSD_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case SSD_ERR_WORKSPACE: return "workspace missing or too small";
        case SSD_ERR_CUDA: return "CUDA error";
        case SSD_ERR_TIMEOUT: return "device wait timed out (outputs invalid)";
        case SSD_ERR_DEVICE: return "device-side check failed (outputs invalid)";
        case SSD_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the built-in array holds";
        default: return "unknown status";
    }
}

extern "C" int ssd_fwd_workspace_size(const ssd_dims *dims, size_t *bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    Problem p;
    int st = check_dims(dims, &p);
    if (st != SSD_OK) return st;
    int32_t path = 0;
    if ((st = choose_path(dims, p, &path)) != SSD_OK) return st;
    *bytes = workspace_for(p, path);
    return SSD_OK;
}

extern "C" int ssd_fwd_path(const ssd_dims *dims, int32_t *path) {
    if (!path) return SSD_ERR_INVALID_ARG;
    Problem p;
    int st = check_dims(dims, &p);
    if (st != SSD_OK) return st;
    return choose_path(dims, p, path);
}

extern "C" int ssd_fwd(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                       const void *B, const void *C, const float *D, const float *init_state,
                       void *y, float *final_state, void *workspace, size_t workspace_bytes,
                       void *stream) {
    Problem p;
    int st = check_dims(dims, &p);
    if (st != SSD_OK) return st;
    int32_t path = 0;
    if ((st = choose_path(dims, p, &path)) != SSD_OK) return st;
    const bool empty = (p.b == 0 || p.T == 0);
    if (!empty && (!x || !dt || !A || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    const void *ptrs[] = {x, dt, A, B, C, D, init_state, y, final_state};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return SSD_ERR_ALIGNMENT;
    if (!empty && y == x) return SSD_ERR_INVALID_ARG;
    const size_t need = workspace_for(p, path);
    if (!workspace || workspace_bytes < need) return SSD_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SSD_ERR_ALIGNMENT;

    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D;
    p.init = init_state; p.y = y; p.final_state = final_state;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t e;
    if (!empty && path == SSD_PATH_TCGEN05) {
        // each clears its own status block (and counters)
        e = diag_supports(p) ? diag_launch(p, workspace, s) : fused_launch(p, workspace, workspace_bytes, s);
    } else {
        e = cudaMemsetAsync(workspace, 0, kStatusBytes, s);
        if (e == cudaSuccess) e = empty ? launch_copy_state(p, s) : generic_launch(p, generic_carve(p, workspace), s);
    }
    return note_cuda(e);
}

// Backward: the gradients of sum y * dy + sum final_state * dfinal (CUDA cores).
static int bwd_check(const ssd_dims *dims, Problem *p) {
    int st = check_dims(dims, p);
    if (st != SSD_OK) return st;
    if (dims->path == SSD_PATH_TCGEN05) return SSD_ERR_UNSUPPORTED;
    return bwd_supports(*p) ? SSD_OK : SSD_ERR_UNSUPPORTED;
}

extern "C" int ssd_bwd_workspace_size(const ssd_dims *dims, size_t *bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    Problem p;
    const int st = bwd_check(dims, &p);
    if (st != SSD_OK) return st;
    *bytes = bwd_workspace_bytes(p, dims->path == SSD_PATH_AUTO);
    return SSD_OK;
}

extern "C" int ssd_bwd(const ssd_dims *dims, const void *x, const float *dt, const float *A, const void *B,
                       const void *C, const float *D, const float *init_state, const void *dy,
                       const float *dfinal, void *dx, float *ddt, float *dA, void *dB, void *dC, float *dD,
                       float *dinit, void *workspace, size_t workspace_bytes, void *stream) {
    Problem p;
    int st = bwd_check(dims, &p);
    if (st != SSD_OK) return st;
    const bool empty = (p.b == 0 || p.T == 0);
    if (!A || (!empty && (!x || !dt || !B || !C || !dy || !dx || !ddt || !dB || !dC)) || !dA)
        return SSD_ERR_INVALID_ARG;
    const void *ptrs[] = {x, dt, A, B, C, D, init_state, dy, dfinal, dx, ddt, dA, dB, dC, dD, dinit};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return SSD_ERR_ALIGNMENT;
    const bool chunked_ok = dims->path == SSD_PATH_AUTO;
    const size_t need = bwd_workspace_bytes(p, chunked_ok);
    if (!workspace || workspace_bytes < need) return SSD_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SSD_ERR_ALIGNMENT;
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.init = init_state;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nA = sizeof(float) * (size_t)(p.a_mode == SSD_A_SCALAR ? p.H : p.H * p.N);
    cudaError_t e;
    if (empty) {
        // no token: dA = dD = 0 and the initial state's gradient is dfinal itself
        const size_t ns = sizeof(float) * (size_t)(p.b * p.H * p.N * p.P);
        e = cudaMemsetAsync(workspace, 0, kStatusBytes, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dA, 0, nA, s);
        if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, sizeof(float) * (size_t)p.H, s);
        if (e == cudaSuccess && dinit && ns)
            e = dfinal ? cudaMemcpyAsync(dinit, dfinal, ns, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(dinit, 0, ns, s);
        return note_cuda(e);
    }
    BwdGrads g{dy, dfinal, dx, ddt, dA, dB, dC, dD, dinit};
    return note_cuda(bwd_launch(p, g, workspace, s, chunked_ok));
}

// The linear form (ssd_scan) and its one-token case (ssd_decode_step): same argument checks as
// ssd_fwd, no workspace.
static int scan_call(const ssd_dims *dims, const void *x, const float *dt, const float *A, const void *B,
                     const void *C, const float *D, const float *init_state, void *y, float *final_state,
                     void *stream) {
    Problem p;
    int st = check_dims(dims, &p);
    if (st != SSD_OK) return st;
    if (dims->path != SSD_PATH_AUTO) return SSD_ERR_INVALID_ARG;
    if (!scan_supports(p)) return SSD_ERR_UNSUPPORTED;
    const bool empty = (p.b == 0 || p.T == 0);
    if (!empty && (!x || !dt || !A || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    // element alignment only (the linear form reads elements one by one): a decode step's
    // token is usually a slice of a larger buffer
    const uintptr_t io_mask = p.io_dtype == SSD_DTYPE_BF16 ? 1u : 3u;
    const void *io_ptrs[] = {x, B, C, y};
    for (const void *q : io_ptrs)
        if (q && (reinterpret_cast<uintptr_t>(q) & io_mask)) return SSD_ERR_ALIGNMENT;
    const void *f32_ptrs[] = {dt, A, D, init_state, final_state};
    for (const void *q : f32_ptrs)
        if (q && (reinterpret_cast<uintptr_t>(q) & 3u)) return SSD_ERR_ALIGNMENT;
    if (!empty && y == x) return SSD_ERR_INVALID_ARG;
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D;
    p.init = init_state; p.y = y; p.final_state = final_state;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (empty) {
        // final_state <- init_state (an in-place state is already there)
        if (!final_state || final_state == init_state) return SSD_OK;
        return note_cuda(launch_copy_state(p, s));
    }
    return note_cuda(scan_launch(p, s));
}

extern "C" int ssd_scan(const ssd_dims *dims, const void *x, const float *dt, const float *A, const void *B,
                        const void *C, const float *D, const float *init_state, void *y, float *final_state,
                        void *stream) {
    return scan_call(dims, x, dt, A, B, C, D, init_state, y, final_state, stream);
}

extern "C" int ssd_decode_step(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                               const void *B, const void *C, const float *D, float *state, void *y,
                               void *stream) {
    if (!dims) return SSD_ERR_INVALID_ARG;
    if (dims->T != 1 || !state) return SSD_ERR_INVALID_ARG;
    return scan_call(dims, x, dt, A, B, C, D, state, y, state, stream);
}

extern "C" int ssd_check_device_status(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < sizeof(int)) return SSD_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return note_cuda(e);
    int word = 0;
    if ((e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return note_cuda(e);
    const int zero = 0;
    if ((e = cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess) return note_cuda(e);
    return word;
}

extern "C" int ssd_debug_set_wait(int64_t spin_limit, int64_t withhold_chunk) {
    g_spin_limit.store(spin_limit);
    g_withhold.store(withhold_chunk);
    return SSD_OK;
}

extern "C" int ssd_debug_set_kernel_events(void *start_event, void *stop_event) {
    g_ev_start.store(start_event);
    g_ev_stop.store(stop_event);
    return SSD_OK;
}

extern "C" const char *ssd_last_cuda_error(void) {
    return cudaGetErrorString(static_cast<cudaError_t>(g_last_cuda.load()));
}

extern "C" int ssd_launch_count(uint64_t *count) {
    if (!count) return SSD_ERR_INVALID_ARG;
    *count = g_launches.load();
    return SSD_OK;
}
