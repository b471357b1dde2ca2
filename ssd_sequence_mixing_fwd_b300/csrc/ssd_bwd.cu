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
// 8-token block (checkpoints), and the reverse sweep recomputes each block's 8
// states from its checkpoint into shared memory before walking it backwards
// (short blocks: four CTAs per SM).
//
// Work split: one CTA per (batch row, head, slice of R = 1024 / P state rows);
// thread t owns state row r = t / (P/W) of the slice and W = 4 consecutive columns,
// so a row's P columns are P/W consecutive lanes of one warp (P <= 128) and the sums
// over p are warp shuffles; 1024 / W = 256 threads.  The sum over n for dx is
// across rows: a warp's rows are summed by shuffles, the warps' sums by
// shared-memory atomics into the block's dx tile, and the tile goes to an fp32
// accumulator once per block (atomics across slices).  Per-token quantities that are summed over heads or over n later (dB,
// dC per head, dlog) go to workspace arrays; small kernels finish the sums and
// convert to the io dtype.
#include <cuda_bf16.h>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kK = 8;        // tokens per checkpoint block
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
__device__ void stage(const BwdParams &p, int bi, int h, int sl, int t0, float *sa, float *sx, float *sB,
                      float *sC, float *sdy) {
    const int g = h / (p.H / p.G);
    const int L = min(kK, p.T - t0);

    for (int i = threadIdx.x; i < kK * p.P; i += blockDim.x) {
        const int k = i / p.P, c = i % p.P;
        const int64_t off = ((int64_t)bi * p.T + t0 + k) * p.H * p.P + (int64_t)h * p.P + c;
        sx[i] = k < L ? ldf(static_cast<const IO *>(p.x), off) : 0.f;
        if (kDy) sdy[i] = k < L ? ldf(static_cast<const IO *>(p.dy), off) : 0.f;
    }
    for (int i = threadIdx.x; i < kK * p.R; i += blockDim.x) {
        const int k = i / p.R, r = i % p.R, n = sl * p.R + r;
        const int64_t off = ((int64_t)bi * p.T + t0 + k) * p.G * p.N + (int64_t)g * p.N + n;
        const bool ok = k < L && n < p.N;
        sB[i] = ok ? ldf(static_cast<const IO *>(p.B), off) : 0.f;
        if (kDy) sC[i] = ok ? ldf(static_cast<const IO *>(p.C), off) : 0.f;
        // the token's decay of this state row
        sa[i] = ok ? expf(decay_log(p, h, n, p.dt[((int64_t)bi * p.T + t0 + k) * p.H + h])) : 0.f;
    }
}

template <int W> __device__ __forceinline__ void ld_w(const float *src, float (&v)[W]) {
#pragma unroll
    for (int j = 0; j < W; j += 4) {
        const float4 f = *reinterpret_cast<const float4 *>(src + j);
        v[j] = f.x; v[j + 1] = f.y; v[j + 2] = f.z; v[j + 3] = f.w;
    }
}
template <int W> __device__ __forceinline__ void st_w(float *dst, const float (&v)[W]) {
#pragma unroll
    for (int j = 0; j < W; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}

// Forward sweep: the state at the start of every kK-token block.
template <typename IO, int W>
__global__ void __launch_bounds__(kElems / W) bwd_ckpt_kernel(BwdParams p) {
    extern __shared__ float sm[];
    float *sx = sm, *sB = sx + kK * p.P, *sa = sB + kK * p.R;
    const int nsl = p.nsl;
    const int sl = blockIdx.x % nsl, s = blockIdx.x / nsl;
    const int bi = s / p.H, h = s % p.H;
    const int tpr = p.P / W, r = threadIdx.x / tpr, p0 = W * (threadIdx.x % tpr);
    const int n = sl * p.R + r;
    const bool live = n < p.N;
    float hs[W];
    if (p.init && live) ld_w<W>(p.init + ((int64_t)s * p.N + n) * p.P + p0, hs);
    else {
#pragma unroll
        for (int j = 0; j < W; ++j) hs[j] = 0.f;
    }
    float *ck = p.ck + ((int64_t)s * nsl + sl) * p.nK * kElems;
    for (int kb = 0; kb < p.nK; ++kb) {
        st_w<W>(ck + (int64_t)kb * kElems + r * p.P + p0, hs);
        __syncthreads();
        stage<IO, false>(p, bi, h, sl, kb * kK, sa, sx, sB, nullptr, nullptr);
        __syncthreads();
        const int L = min(kK, p.T - kb * kK);
#pragma unroll 4
        for (int k = 0; k < L; ++k) {
            const float a = sa[k * p.R + r];
            const float bn = sB[k * p.R + r];
            float xv[W];
            ld_w<W>(sx + k * p.P + p0, xv);
#pragma unroll
            for (int j = 0; j < W; ++j) hs[j] = fmaf(a, hs[j], bn * xv[j]);
        }
    }
}

// Reverse sweep.
template <typename IO, int W>
__global__ void __launch_bounds__(kElems / W) bwd_reverse_kernel(BwdParams p) {
    extern __shared__ float sm[];
    float *hb = sm;                               // [kK + 1][kElems]: h_{t0-1} .. h_{t0+kK-1}
    float *sx = hb + (kK + 1) * kElems;           // [kK][P]
    float *sdy = sx + kK * p.P;                   // [kK][P]
    float *sB = sdy + kK * p.P;                   // [kK][R]
    float *sC = sB + kK * p.R;                    // [kK][R]
    float *sa = sC + kK * p.R;                    // [kK][R] decays
    float *red = sa + kK * p.R;                   // [kK][P] the block's dx over this slice's rows
    const int nsl = p.nsl;
    const int sl = blockIdx.x % nsl, s = blockIdx.x / nsl;
    const int bi = s / p.H, h = s % p.H;
    const int tpr = p.P / W, r = threadIdx.x / tpr, p0 = W * (threadIdx.x % tpr);
    const int n = sl * p.R + r;
    const bool live = n < p.N;
    float gr[W];
    if (p.dfinal && live) ld_w<W>(p.dfinal + ((int64_t)s * p.N + n) * p.P + p0, gr);
    else {
#pragma unroll
        for (int j = 0; j < W; ++j) gr[j] = 0.f;
    }
    const float *ck = p.ck + ((int64_t)s * nsl + sl) * p.nK * kElems;
    for (int kb = p.nK - 1; kb >= 0; --kb) {
        const int t0 = kb * kK, L = min(kK, p.T - t0);
        __syncthreads();
        stage<IO, true>(p, bi, h, sl, t0, sa, sx, sB, sC, sdy);
        for (int i = threadIdx.x; i < kK * p.P; i += blockDim.x) red[i] = 0.f;
        float hs[W];
        ld_w<W>(ck + (int64_t)kb * kElems + r * p.P + p0, hs);
        __syncthreads();
        st_w<W>(hb + r * p.P + p0, hs);
#pragma unroll 4
        for (int k = 0; k < L; ++k) {
            const float a = sa[k * p.R + r];
            const float bn = sB[k * p.R + r];
            float xv[W];
            ld_w<W>(sx + k * p.P + p0, xv);
#pragma unroll
            for (int j = 0; j < W; ++j) hs[j] = fmaf(a, hs[j], bn * xv[j]);
            st_w<W>(hb + (k + 1) * kElems + r * p.P + p0, hs);
        }
#pragma unroll 2
        for (int k = L - 1; k >= 0; --k) {
            const int t = t0 + k;
            const float a = sa[k * p.R + r];
            const float cn = sC[k * p.R + r], bn = sB[k * p.R + r];
            float hcv[W], hpv[W], dyv[W], xv[W];
            ld_w<W>(hb + (k + 1) * kElems + r * p.P + p0, hcv);
            ld_w<W>(hb + k * kElems + r * p.P + p0, hpv);
            ld_w<W>(sdy + k * p.P + p0, dyv);
            ld_w<W>(sx + k * p.P + p0, xv);
            float c = 0.f, b = 0.f, l = 0.f, xs[W];
#pragma unroll
            for (int j = 0; j < W; ++j) {
                gr[j] = fmaf(cn, dyv[j], gr[j]);
                c = fmaf(hcv[j], dyv[j], c);
                b = fmaf(gr[j], xv[j], b);
                l = fmaf(gr[j], hpv[j], l);
                xs[j] = bn * gr[j];
            }
            // dx over this slice's rows: the warp's rows (lanes tpr apart hold the same columns)
            // by shuffles, the warps by shared-memory atomics
            for (int o = tpr; o < 32; o <<= 1) {
#pragma unroll
                for (int j = 0; j < W; ++j) xs[j] += __shfl_xor_sync(0xffffffffu, xs[j], o);
            }
            if ((threadIdx.x & 31) < tpr) {
#pragma unroll
                for (int j = 0; j < W; ++j) atomicAdd(red + k * p.P + p0 + j, xs[j]);
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
#pragma unroll
            for (int j = 0; j < W; ++j) gr[j] *= a;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < L * p.P; i += blockDim.x) {
            const int k = i / p.P, c2 = i % p.P;
            atomicAdd(p.dxa + (((int64_t)bi * p.T + t0 + k) * p.H + h) * p.P + c2, red[i]);
        }
    }
    if (p.dinit && live) st_w<W>(p.dinit + ((int64_t)s * p.N + n) * p.P + p0, gr);
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
// CTA (head, state row or 0, chunk of kChunk tokens), a block-wide sum added atomically into the
// zeroed outputs.
constexpr int kChunk = 1024;
template <typename IO>
__global__ void __launch_bounds__(256) bwd_finish_params(BwdParams p) {
    __shared__ float part[2][8];
    const int h = blockIdx.x, k = blockIdx.y;     // k: state row (diagonal A), else 0
    float sa = 0.f, sd = 0.f;
    const int64_t nbt = (int64_t)p.b * p.T;
    const int64_t b0 = (int64_t)blockIdx.z * kChunk, b1 = min(nbt, b0 + kChunk);
    for (int64_t bt = b0 + threadIdx.x; bt < b1; bt += blockDim.x) {
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
        for (int w = 0; w < 8; ++w) {
            a += part[0][w];
            d += part[1][w];
        }
        atomicAdd(p.dA + (p.diag ? (int64_t)h * p.N + k : h), a);
        if (k == 0 && p.dD) atomicAdd(p.dD + h, d);
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
    return sizeof(float) * ((size_t)(kK + 1) * kElems + 3 * kK * p.P + 3 * kK * l.R);
}

template <typename IO, int W>
cudaError_t launch_sweeps(const Problem &p, const BwdParams &bp, const BwdLayout &l, cudaStream_t s) {
    const size_t sm_ck = sizeof(float) * (size_t)(kK * p.P + 2 * kK * l.R);
    const size_t sm_rev = reverse_smem(p, l);
    cudaError_t e = cudaFuncSetAttribute(bwd_reverse_kernel<IO, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_rev);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.b * p.H * l.nsl);
    record_dominant_start(s);
    bwd_ckpt_kernel<IO, W><<<grid, kElems / W, sm_ck, s>>>(bp);
    bwd_reverse_kernel<IO, W><<<grid, kElems / W, sm_rev, s>>>(bp);
    record_dominant_stop(s);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_all(const Problem &p, const BwdParams &bp, const BwdLayout &l, cudaStream_t s) {
    // four columns per thread (256 threads): eight (128 threads) measured slower -- fewer warps to
    // hide the per-token latency
    cudaError_t e = launch_sweeps<IO, 4>(p, bp, l, s);
    if (e != cudaSuccess) return e;
    bwd_finish_tokens<IO><<<1184, 256, 0, s>>>(bp);
    bwd_finish_bc<IO><<<1184, 256, 0, s>>>(bp);
    const unsigned chunks = (unsigned)((p.b * p.T + kChunk - 1) / kChunk);
    bwd_finish_params<IO><<<dim3((unsigned)p.H, bp.diag ? (unsigned)p.N : 1u, chunks), 256, 0, s>>>(bp);
    note_launches(5);
    return cudaGetLastError();
}

}  // namespace

bool bwd_supports(const Problem &p) {
    if (p.P < 4 || p.P > 128 || (p.P & (p.P - 1))) return false;   // a state row's columns within one warp
    if ((p.b * p.T + kChunk - 1) / kChunk > 65535) return false;     // grid z of the parameter sums
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
    if (e == cudaSuccess)
        e = cudaMemsetAsync(gr.dA, 0, sizeof(float) * (size_t)(p.a_mode == SSD_A_SCALAR ? p.H : p.H * p.N), s);
    if (e == cudaSuccess && gr.dD) e = cudaMemsetAsync(gr.dD, 0, sizeof(float) * (size_t)p.H, s);
    if (e != cudaSuccess) return e;
    return p.io_dtype == SSD_DTYPE_BF16 ? launch_all<__nv_bfloat16>(p, bp, l, s) : launch_all<float>(p, bp, l, s);
}

}  // namespace ssd
