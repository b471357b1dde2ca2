// ssd_bwd.cu -- backward of the SSD forward pass on CUDA cores (fp32).
//
// The gradients of L = sum y * dy + sum final_state * dfinal with respect to x,
// dt, A, B, C, D and init_state, for the map ssd_fwd computes (Structured State
// Space Duality, "The recurrence as one matrix"; the pages frame the chunked
// algorithm around training cost -- "The chunked algorithm takes both" -- but
// give no backward, so this is the chain rule of the recurrence).  With
// g_t = dL/dh_t, running from dfinal backwards,
//
//   g   += C_t dy_t^T             dC_t += h_t dy_t        dx_t = g^T B_t + D dy_t
//   dB_t += g x_t                 dlog_t = a_t o rowsum(g o h_{t-1})
//   ddt_t = sum_n A_n dlog_t[n]   dA += dt_t dlog_t       g = a_t o g
//
// and dinit = g after the first token (the sums over p are per state row; dB,
// dC, dA and dD are summed over the heads / batch rows that share them).  The
// reverse sweep needs h_t and h_{t-1} at every token, so the states are
// recomputed: a forward sweep stores the state at the start of every
// 32-token block (checkpoints), and the reverse sweep recomputes each block's 32
// states from its checkpoint into shared memory before walking it backwards.
//
// Work split: one CTA per (batch row, head, slice of R = 1024 / P state rows), 256
// threads; thread t owns state row r = t / (P/4) of the slice and columns
// 4 (t mod P/4) .. + 3, so a row's P columns are P/4 consecutive lanes of one warp
// (P <= 128) and the sums over p are warp shuffles.  The sum over n for dx is
// across rows: through shared memory within the CTA and fp32 atomics across
// slices.  Per-token quantities that are summed over heads or over n later (dB,
// dC per head, dlog) go to workspace arrays; small kernels finish the sums and
// convert to the io dtype.
#include <cuda_bf16.h>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kT = 256;      // threads per CTA
constexpr int kK = 32;       // tokens per checkpoint block
constexpr int kElems = 1024; // state entries per CTA (R rows x P columns)

template <typename IO> __device__ __forceinline__ float ldf(const IO *p, int64_t i);
template <> __device__ __forceinline__ float ldf<float>(const float *p, int64_t i) { return p[i]; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
template <typename IO> __device__ __forceinline__ void stf(IO *p, int64_t i, float v);
template <> __device__ __forceinline__ void stf<float>(float *p, int64_t i, float v) { p[i] = v; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

struct BwdParams {
    const void *x, *B, *C, *dy;
    const float *dt, *A, *D, *init, *dfinal;
    void *dx, *dB, *dC;
    float *ddt, *dA, *dD, *dinit;
    float *ck;       // (b, H, nsl, nK, R, P) checkpoints
    float *dBh;      // (b, T, H, N) per-head dB
    float *dCh;      // (b, T, H, N) per-head dC
    float *dl;       // (b, T, H, N) dlog
    float *dxa;      // (b, T, H, P) dx accumulator (fp32, atomics over slices)
    int b, T, H, P, N, G, R, nsl, nK, diag;
};

__device__ __forceinline__ float decay_log(const BwdParams &p, int h, int n, float dtv) {
    return dtv * (p.diag ? p.A[(int64_t)h * p.N + n] : p.A[h]);
}

// Stage kK tokens of one (batch row, head, slice): dt, x, B and C rows of the slice (and dy).
template <typename IO, bool kDy>
__device__ void stage(const BwdParams &p, int bi, int h, int sl, int t0, float *sdt, float *sx, float *sB,
                      float *sC, float *sdy) {
    const int g = h / (p.H / p.G);
    const int L = min(kK, p.T - t0);
    for (int i = threadIdx.x; i < kK; i += kT)
        sdt[i] = i < L ? p.dt[((int64_t)bi * p.T + t0 + i) * p.H + h] : 0.f;
    for (int i = threadIdx.x; i < kK * p.P; i += kT) {
        const int k = i / p.P, c = i % p.P;
        const int64_t off = ((int64_t)bi * p.T + t0 + k) * p.H * p.P + (int64_t)h * p.P + c;
        sx[i] = k < L ? ldf(static_cast<const IO *>(p.x), off) : 0.f;
        if (kDy) sdy[i] = k < L ? ldf(static_cast<const IO *>(p.dy), off) : 0.f;
    }
    for (int i = threadIdx.x; i < kK * p.R; i += kT) {
        const int k = i / p.R, r = i % p.R, n = sl * p.R + r;
        const int64_t off = ((int64_t)bi * p.T + t0 + k) * p.G * p.N + (int64_t)g * p.N + n;
        const bool ok = k < L && n < p.N;
        sB[i] = ok ? ldf(static_cast<const IO *>(p.B), off) : 0.f;
        if (kDy) sC[i] = ok ? ldf(static_cast<const IO *>(p.C), off) : 0.f;
    }
}

// Forward sweep: the state at the start of every kK-token block.
template <typename IO>
__global__ void __launch_bounds__(kT) bwd_ckpt_kernel(BwdParams p) {
    __shared__ float sdt[kK];
    extern __shared__ float sm[];
    float *sx = sm, *sB = sx + kK * p.P;
    const int nsl = p.nsl;
    const int sl = blockIdx.x % nsl, s = blockIdx.x / nsl;
    const int bi = s / p.H, h = s % p.H;
    const int tpr = p.P / 4, r = threadIdx.x / tpr, p0 = 4 * (threadIdx.x % tpr);
    const int n = sl * p.R + r;
    const bool live = n < p.N;
    float hs[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        hs[j] = (p.init && live) ? p.init[((int64_t)s * p.N + n) * p.P + p0 + j] : 0.f;
    float *ck = p.ck + ((int64_t)s * nsl + sl) * p.nK * kElems;
    for (int kb = 0; kb < p.nK; ++kb) {
        *reinterpret_cast<float4 *>(ck + (int64_t)kb * kElems + r * p.P + p0) = make_float4(hs[0], hs[1], hs[2], hs[3]);
        __syncthreads();
        stage<IO, false>(p, bi, h, sl, kb * kK, sdt, sx, sB, nullptr, nullptr);
        __syncthreads();
        const int L = min(kK, p.T - kb * kK);
        for (int k = 0; k < L; ++k) {
            const float a = live ? expf(decay_log(p, h, n, sdt[k])) : 0.f;
            const float bn = sB[k * p.R + r];
#pragma unroll
            for (int j = 0; j < 4; ++j) hs[j] = fmaf(a, hs[j], bn * sx[k * p.P + p0 + j]);
        }
    }
}

// Reverse sweep.
template <typename IO>
__global__ void __launch_bounds__(kT) bwd_reverse_kernel(BwdParams p) {
    __shared__ float sdt[kK];
    extern __shared__ float sm[];
    float *hb = sm;                               // [kK + 1][kElems]: h_{t0-1} .. h_{t0+kK-1}
    float *sx = hb + (kK + 1) * kElems;           // [kK][P]
    float *sdy = sx + kK * p.P;                   // [kK][P]
    float *sB = sdy + kK * p.P;                   // [kK][R]
    float *sC = sB + kK * p.R;                    // [kK][R]
    float *red = sC + kK * p.R;                   // [R][P] partial dx
    const int nsl = p.nsl;
    const int sl = blockIdx.x % nsl, s = blockIdx.x / nsl;
    const int bi = s / p.H, h = s % p.H;
    const int tpr = p.P / 4, r = threadIdx.x / tpr, p0 = 4 * (threadIdx.x % tpr);
    const int n = sl * p.R + r;
    const bool live = n < p.N;
    float gr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        gr[j] = (p.dfinal && live) ? p.dfinal[((int64_t)s * p.N + n) * p.P + p0 + j] : 0.f;
    const float *ck = p.ck + ((int64_t)s * nsl + sl) * p.nK * kElems;
    for (int kb = p.nK - 1; kb >= 0; --kb) {
        const int t0 = kb * kK, L = min(kK, p.T - t0);
        __syncthreads();
        stage<IO, true>(p, bi, h, sl, t0, sdt, sx, sB, sC, sdy);
        float hs[4];
        {
            const float4 v = *reinterpret_cast<const float4 *>(ck + (int64_t)kb * kElems + r * p.P + p0);
            hs[0] = v.x; hs[1] = v.y; hs[2] = v.z; hs[3] = v.w;
        }
        __syncthreads();
        *reinterpret_cast<float4 *>(hb + r * p.P + p0) = make_float4(hs[0], hs[1], hs[2], hs[3]);
        for (int k = 0; k < L; ++k) {
            const float a = live ? expf(decay_log(p, h, n, sdt[k])) : 0.f;
            const float bn = sB[k * p.R + r];
#pragma unroll
            for (int j = 0; j < 4; ++j) hs[j] = fmaf(a, hs[j], bn * sx[k * p.P + p0 + j]);
            *reinterpret_cast<float4 *>(hb + (k + 1) * kElems + r * p.P + p0) = make_float4(hs[0], hs[1], hs[2], hs[3]);
        }
        for (int k = L - 1; k >= 0; --k) {
            const int t = t0 + k;
            const float a = live ? expf(decay_log(p, h, n, sdt[k])) : 0.f;
            const float cn = sC[k * p.R + r], bn = sB[k * p.R + r];
            const float4 hc = *reinterpret_cast<const float4 *>(hb + (k + 1) * kElems + r * p.P + p0);
            const float4 hp = *reinterpret_cast<const float4 *>(hb + k * kElems + r * p.P + p0);
            const float hcv[4] = {hc.x, hc.y, hc.z, hc.w}, hpv[4] = {hp.x, hp.y, hp.z, hp.w};
            float c = 0.f, b = 0.f, l = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float dyv = sdy[k * p.P + p0 + j];
                gr[j] = fmaf(cn, dyv, gr[j]);
                c = fmaf(hcv[j], dyv, c);
                b = fmaf(gr[j], sx[k * p.P + p0 + j], b);
                l = fmaf(gr[j], hpv[j], l);
                red[r * p.P + p0 + j] = bn * gr[j];
            }
            // (offsets below tpr stay inside the row's aligned group of tpr lanes)
            for (int o = tpr >> 1; o >= 1; o >>= 1) {
                c += __shfl_xor_sync(0xffffffffu, c, o);
                b += __shfl_xor_sync(0xffffffffu, b, o);
                l += __shfl_xor_sync(0xffffffffu, l, o);
            }
            if (p0 == 0 && live) {
                const int64_t o = (((int64_t)bi * p.T + t) * p.H + h) * p.N + n;
                p.dCh[o] = c;
                p.dBh[o] = b;
                p.dl[o] = a * l;
            }
            __syncthreads();
            for (int c2 = threadIdx.x; c2 < p.P; c2 += kT) {
                float acc = 0.f;
                for (int rr = 0; rr < p.R; ++rr) acc += red[rr * p.P + c2];
                atomicAdd(p.dxa + (((int64_t)bi * p.T + t) * p.H + h) * p.P + c2, acc);
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 4; ++j) gr[j] *= a;
        }
    }
    if (p.dinit && live)
        *reinterpret_cast<float4 *>(p.dinit + ((int64_t)s * p.N + n) * p.P + p0) = make_float4(gr[0], gr[1], gr[2], gr[3]);
}

// dx = accumulated sum (+ D dy) in the io dtype; ddt = sum_n A_n dlog.
template <typename IO>
__global__ void bwd_finish_tokens(BwdParams p) {
    const int64_t ntok = (int64_t)p.b * p.T * p.H;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ntok * p.P; i += (int64_t)gridDim.x * blockDim.x) {
        const int h = (int)((i / p.P) % p.H);
        float v = p.dxa[i];
        if (p.D) v = fmaf(p.D[h], ldf(static_cast<const IO *>(p.dy), i), v);
        stf(static_cast<IO *>(p.dx), i, v);
    }
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ntok; i += (int64_t)gridDim.x * blockDim.x) {
        const int h = (int)(i % p.H);
        const float *dl = p.dl + i * p.N;
        float acc = 0.f;
        for (int n = 0; n < p.N; ++n) acc = fmaf(p.diag ? p.A[(int64_t)h * p.N + n] : 1.f, dl[n], acc);
        p.ddt[i] = p.diag ? acc : acc * p.A[h];
    }
}

// dB, dC: sums over the heads of a group, in the io dtype.
template <typename IO>
__global__ void bwd_finish_bc(BwdParams p) {
    const int hpg = p.H / p.G;
    const int64_t tot = (int64_t)p.b * p.T * p.G * p.N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < tot; i += (int64_t)gridDim.x * blockDim.x) {
        const int n = (int)(i % p.N);
        const int g = (int)((i / p.N) % p.G);
        const int64_t bt = i / ((int64_t)p.N * p.G);
        float sb = 0.f, sc = 0.f;
        for (int h = g * hpg; h < (g + 1) * hpg; ++h) {
            const int64_t o = (bt * p.H + h) * p.N + n;
            sb += p.dBh[o];
            sc += p.dCh[o];
        }
        stf(static_cast<IO *>(p.dB), i, sb);
        stf(static_cast<IO *>(p.dC), i, sc);
    }
}

// dA (sum over batch rows and tokens of dt dlog; over n too for scalar A) and dD (sum of dy x):
// one CTA per head and (diagonal A) per state row, a block-wide reduction.
template <typename IO>
__global__ void bwd_finish_params(BwdParams p) {
    __shared__ float part[2][kT / 32];
    const int h = blockIdx.x, k = blockIdx.y;     // k: state row (diagonal A), else 0
    float sa = 0.f, sd = 0.f;
    const int64_t nbt = (int64_t)p.b * p.T;
    for (int64_t bt = threadIdx.x; bt < nbt; bt += blockDim.x) {
        const int64_t tok = bt * p.H + h;
        const float dtv = p.dt[tok];
        if (p.diag) {
            sa = fmaf(dtv, p.dl[tok * p.N + k], sa);
        } else {
            float l = 0.f;
            for (int n = 0; n < p.N; ++n) l += p.dl[tok * p.N + n];
            sa = fmaf(dtv, l, sa);
        }
        if (k == 0 && p.dD)
            for (int c = 0; c < p.P; ++c)
                sd = fmaf(ldf(static_cast<const IO *>(p.dy), tok * p.P + c), ldf(static_cast<const IO *>(p.x), tok * p.P + c), sd);
    }
    for (int o = 16; o >= 1; o >>= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
    }
    if ((threadIdx.x & 31) == 0) {
        part[0][threadIdx.x >> 5] = sa;
        part[1][threadIdx.x >> 5] = sd;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f, d = 0.f;
        for (int w = 0; w < kT / 32; ++w) {
            a += part[0][w];
            d += part[1][w];
        }
        p.dA[p.diag ? (int64_t)h * p.N + k : h] = a;
        if (k == 0 && p.dD) p.dD[h] = d;
    }
}

struct BwdLayout {
    int R, nsl, nK;
    size_t off_ck, off_dbh, off_dch, off_dl, off_dxa, total;
};

BwdLayout bwd_layout(const Problem &p) {
    BwdLayout l;
    l.R = kElems / (int)p.P;
    l.nsl = (int)((p.N + l.R - 1) / l.R);
    l.nK = (int)((p.T + kK - 1) / kK);
    const size_t tokh = (size_t)(p.b * p.T * p.H);
    l.off_ck = kStatusBytes;
    l.off_dbh = align_up(l.off_ck + sizeof(float) * (size_t)(p.b * p.H) * l.nsl * l.nK * kElems, 256);
    l.off_dch = align_up(l.off_dbh + sizeof(float) * tokh * p.N, 256);
    l.off_dl = align_up(l.off_dch + sizeof(float) * tokh * p.N, 256);
    l.off_dxa = align_up(l.off_dl + sizeof(float) * tokh * p.N, 256);
    l.total = align_up(l.off_dxa + sizeof(float) * tokh * p.P, 256);
    return l;
}

size_t reverse_smem(const Problem &p, const BwdLayout &l) {
    return sizeof(float) * ((size_t)(kK + 1) * kElems + 2 * kK * p.P + 2 * kK * l.R + (size_t)l.R * p.P);
}

template <typename IO>
cudaError_t launch_all(const Problem &p, const BwdParams &bp, const BwdLayout &l, cudaStream_t s) {
    const size_t sm_ck = sizeof(float) * (size_t)(kK * p.P + kK * l.R);
    const size_t sm_rev = reverse_smem(p, l);
    cudaError_t e = cudaFuncSetAttribute(bwd_reverse_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_rev);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.H * l.nsl);
    record_dominant_start(s);
    bwd_ckpt_kernel<IO><<<grid, kT, sm_ck, s>>>(bp);
    bwd_reverse_kernel<IO><<<grid, kT, sm_rev, s>>>(bp);
    record_dominant_stop(s);
    bwd_finish_tokens<IO><<<1184, 256, 0, s>>>(bp);
    bwd_finish_bc<IO><<<1184, 256, 0, s>>>(bp);
    bwd_finish_params<IO><<<dim3((unsigned)p.H, bp.diag ? (unsigned)p.N : 1u), kT, 0, s>>>(bp);
    note_launches(5);
    return cudaGetLastError();
}

}  // namespace

bool bwd_supports(const Problem &p) {
    if (p.P < 4 || p.P > 128 || (p.P & (p.P - 1))) return false;   // a state row's columns within one warp
    if (p.b * p.H * ((p.N + kElems / p.P - 1) / (kElems / p.P)) > (int64_t)INT32_MAX) return false;
    if (p.T > (int64_t)INT32_MAX / 2) return false;
    return true;
}

size_t bwd_workspace_bytes(const Problem &p) { return bwd_layout(p).total; }

cudaError_t bwd_launch(const Problem &p, const BwdGrads &gr, void *ws, cudaStream_t s) {
    const BwdLayout l = bwd_layout(p);
    char *base = static_cast<char *>(ws);
    BwdParams bp;
    bp.x = p.x; bp.B = p.B; bp.C = p.C; bp.dy = gr.dy;
    bp.dt = p.dt; bp.A = p.A; bp.D = p.D; bp.init = p.init; bp.dfinal = gr.dfinal;
    bp.dx = gr.dx; bp.dB = gr.dB; bp.dC = gr.dC;
    bp.ddt = gr.ddt; bp.dA = gr.dA; bp.dD = gr.dD; bp.dinit = gr.dinit;
    bp.ck = reinterpret_cast<float *>(base + l.off_ck);
    bp.dBh = reinterpret_cast<float *>(base + l.off_dbh);
    bp.dCh = reinterpret_cast<float *>(base + l.off_dch);
    bp.dl = reinterpret_cast<float *>(base + l.off_dl);
    bp.dxa = reinterpret_cast<float *>(base + l.off_dxa);
    bp.b = (int)p.b; bp.T = (int)p.T; bp.H = (int)p.H; bp.P = (int)p.P; bp.N = (int)p.N; bp.G = (int)p.G;
    bp.R = l.R; bp.nsl = l.nsl; bp.nK = l.nK;
    bp.diag = p.a_mode == SSD_A_DIAGONAL;
    cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(bp.dxa, 0, sizeof(float) * (size_t)(p.b * p.T * p.H * p.P), s);
    if (e != cudaSuccess) return e;
    return p.io_dtype == SSD_DTYPE_BF16 ? launch_all<__nv_bfloat16>(p, bp, l, s) : launch_all<float>(p, bp, l, s);
}

}  // namespace ssd
