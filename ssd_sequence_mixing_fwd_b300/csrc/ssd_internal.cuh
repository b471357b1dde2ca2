// ssd_internal.cuh -- shared host/device definitions of libssd_b300.
//
// Internal to the library; the public boundary is include/ssd.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ssd.h"

namespace ssd {

// One validated call, as the kernels see it.  Shapes and layouts are those of
// include/ssd.h; nc = ceil(T / Q) chunks per sequence.
struct Problem {
    int64_t b, T, H, P, N, G, Q, nc;
    int a_mode;      // SSD_A_SCALAR / SSD_A_DIAGONAL
    int io_dtype;    // SSD_DTYPE_BF16 / SSD_DTYPE_F32
    const void *x;
    const float *dt;
    const float *A;
    const void *B;
    const void *C;
    const float *D;
    const float *init;
    void *y;
    float *final_state;
};

// Device-side status word: the first 4 bytes of every workspace.
constexpr size_t kStatusBytes = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---- generic CUDA-core path (csrc/ssd_generic.cu) -------------------------
// Workspace: [status | chunk_sum (b,H,nc) f32 | states (b,H,nc,N,P) f32].
struct GenericWorkspace {
    int *status;
    float *chunk_sum;
    float *states;
};
size_t generic_workspace_bytes(const Problem &p);
GenericWorkspace generic_carve(const Problem &p, void *ws);
bool generic_supports(const Problem &p);
cudaError_t generic_launch(const Problem &p, const GenericWorkspace &w, cudaStream_t s);
// the state passing alone: w.states holds every chunk's state s_c and w.chunk_sum its summed
// log decay; leaves the state entering each chunk in place (p.final_state written when set)
cudaError_t generic_passing_launch(const Problem &p, const GenericWorkspace &w, cudaStream_t s);

// ---- fused tcgen05 path (csrc/ssd_fused_tc.cu) ----------------------------
size_t fused_workspace_bytes(const Problem &p);
bool fused_supports(const Problem &p);
cudaError_t fused_launch(const Problem &p, void *ws, size_t ws_bytes, cudaStream_t s);

// ---- diagonal-A tcgen05 path (csrc/ssd_diag_tc.cu); workspace: the status block
bool diag_supports(const Problem &p);
size_t diag_workspace_bytes(const Problem &p);
cudaError_t diag_launch(const Problem &p, void *ws, cudaStream_t s);

// ---- backward (csrc/ssd_bwd.cu): gradient buffers of one call
struct BwdGrads {
    const void *dy;        // (b,T,H,P) io dtype
    const float *dfinal;   // (b,H,N,P) or null
    void *dx;              // (b,T,H,P) io dtype
    float *ddt;            // (b,T,H)
    float *dA;             // like A
    void *dB, *dC;         // (b,T,G,N) io dtype
    float *dD;             // (H) or null
    float *dinit;          // (b,H,N,P) or null
};
bool bwd_supports(const Problem &p);
// chunked_ok: the chunked path may be taken where it applies (SSD_PATH_AUTO); else the
// token recurrence runs
size_t bwd_workspace_bytes(const Problem &p, bool chunked_ok);
cudaError_t bwd_launch(const Problem &p, const BwdGrads &g, void *ws, cudaStream_t s, bool chunked_ok);

// ---- linear-form scan (csrc/ssd_scan.cu): no workspace ---------------------
bool scan_supports(const Problem &p);
cudaError_t scan_launch(const Problem &p, cudaStream_t s);

// ---- small helpers (csrc/ssd_api.cu) --------------------------------------
// Host-side validation of ssd_dims shared by the entry points (fills *prob).
int validate_dims(const ssd_dims *d, Problem *prob);
// final_state <- init_state (or zero) for T == 0.
cudaError_t launch_copy_state(const Problem &p, cudaStream_t s);

// Test hook values (ssd_debug_set_wait).
int64_t debug_spin_limit();
int64_t debug_withhold_chunk();

// Measurement hooks: count launches; bracket the dominant kernel with the
// caller's events when set (ssd_debug_set_kernel_events).
void note_launches(int n);
// Records a failed CUDA call for ssd_last_cuda_error; returns SSD_OK or SSD_ERR_CUDA.
int note_cuda(cudaError_t e);
void record_dominant_start(cudaStream_t s);
void record_dominant_stop(cudaStream_t s);

}  // namespace ssd
