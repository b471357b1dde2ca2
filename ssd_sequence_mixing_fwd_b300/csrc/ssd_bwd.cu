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

#include <cstring>

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

// ---- chunked backward (scalar A) ---------------------------------------------------
// The same gradients, chunk by chunk as dense products: the chunked algorithm of
// Structured State Space Duality, "The chunked algorithm takes both", run backwards (the
// quadratic form inside each chunk, the state between chunks), which replaces the
// per-token sums of the reverse sweep (one over p per state row, one over n per column:
// shuffles and shared-memory atomics at every token) with products over whole chunks.
// With Q-token chunks, cum the in-chunk prefix sum of dt A, L_ij = e^{cum_i - cum_j}
// (j <= i, else 0), w_j = e^{cum_Q - cum_j}, e_i = e^{cum_i} (all <= 1), h the state
// entering the chunk and g = dL/dh at its end:
//   S = L o (C B^T),  G = L o (dY X^T)
//   dX = S^T dY + w o (B g) + D dY
//   dC = G B + e o (dY h^T),  dB = G^T C + w o (X g^T)
//   the adjoint entering the chunk: e^{cum_Q} g + C^T (e o dY)
//   with K = G o (C B^T), v_j = x_j.(B g)_j and u_i = C_i.(h dY_i), the gradient with respect
//   to the in-chunk prefix sums, summed over i >= k, is
//     rc_k = e^{cum_Q} <g, h> + sum_{j<k} w_j v_j + sum_{i>=k, j<k} K_ij + sum_{i>=k} e_i u_i
//   (the pairs of K with both indices >= k, and the w v terms of tokens >= k, cancel exactly
//   and are left out rather than summed and subtracted: at fp32 that difference lost a
//   decade of dA's digits), and ddt_k = A rc_k, dA += sum_k dt_k rc_k.
// Kernels: bwd_chunk_cb forms C B^T once per chunk and B/C group (all the group's heads
// share it); bwd_chunk_sr forms each chunk's state B^T (w o X) and C^T (e o dY); the
// generic forward's state passing turns the states into the state entering every chunk;
// bwd_state_reverse runs the adjoint backwards over the chunks (each chunk's end adjoint
// left in place, and dinit); bwd_chunk_grad does the rest, one CTA per chunk and head,
// every product in exact fp32 on the CUDA cores.
// shared-memory floats of the product kernel (bwd_chunk_grad) for Q-token chunks
constexpr size_t grad_floats(int N, int P, int Q) {
    return 8 + (size_t)2 * Q * (P + 1) + 2 * Q * (N + 1) + 2 * N * (P + 1) + 3 * Q * (Q + 1) + 5 * Q;
}
constexpr size_t kSmemFloats = 227 * 1024 / 4;
// tokens per chunk: 64 where the product kernel's shared memory fits, else 32 (0: neither)
constexpr int chunk_len_of(int N, int P) {
    return grad_floats(N, P, 64) <= kSmemFloats ? 64 : grad_floats(N, P, 32) <= kSmemFloats ? 32 : 0;
}
template <int N, int P> constexpr int chunk_len() { return chunk_len_of(N, P); }
constexpr int kCT = 256;          // threads of the chunk kernels

struct BwdCParams {
    const void *x, *B, *C, *dy;
    const float *dt, *A, *D, *dfinal;
    void *dx;
    float *ddt, *dA, *dD, *dinit;
    float *states;         // (b, H, nc, N, P): each chunk's state, then the state entering it
    float *csum;           // (b, H, nc): sum of dt A over each chunk
    float *gst;            // (b, H, nc, N, P): C^T (e o dY), then the adjoint at each chunk's end
    float *dBh, *dCh;      // (b, T, H, N) per head
    float *cbg;            // (b, nc, G, Q, Q): C B^T of each chunk and B/C group
    int b, T, H, G, N, P, nc;
};

// cum[0..Q): inclusive prefix sum of dt A over the chunk (dt of token k at dt[k * stride];
// zero past L, so the sum holds its last value there).  All threads of the block.
template <int Q>
__device__ __forceinline__ void chunk_cum(const float *dt, int64_t stride, float Ah, int L, float *cum) {
    if (threadIdx.x < Q) {
        const int i = threadIdx.x;
        float v = i < L ? dt[i * stride] * Ah : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if ((i & 31) >= o) v += u;
        }
        cum[i] = v;
    }
    __syncthreads();
    if (threadIdx.x >= 32 && threadIdx.x < Q) cum[threadIdx.x] += cum[31];
    __syncthreads();
}

// 16 bytes of io values as fp32
__device__ __forceinline__ void unpack16(const uint4 &u, const float *, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4 &u, const __nv_bfloat16 *, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// dst[k * ds + c] = scale_k * src[base + k * rs + c] (fp32) for k < valid, 0 past valid, over a
// ROWS x COLS tile: every thread issues all of its 16-byte loads before its first store (the
// rows start on 16-byte boundaries: COLS, rs and base are multiples of the 16-byte vector)
template <typename IO, int ROWS, int COLS>
__device__ __forceinline__ void load_tile(float *dst, int ds, const IO *src, int64_t base, int64_t rs, int valid,
                                          const float *scale = nullptr) {
    constexpr int V = 16 / sizeof(IO);
    constexpr int NV = ROWS * COLS / V;
    constexpr int PER = (NV + kCT - 1) / kCT;
    static_assert(COLS % V == 0, "tile rows are whole 16-byte vectors");
    uint4 buf[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int e = threadIdx.x + u * kCT;
        const int k = (e * V) / COLS, c = (e * V) % COLS;
        buf[u] = make_uint4(0u, 0u, 0u, 0u);
        if (e < NV && k < valid) buf[u] = __ldg(reinterpret_cast<const uint4 *>(src + base + (int64_t)k * rs + c));
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int e = threadIdx.x + u * kCT;
        if (e < NV) {
            const int k = (e * V) / COLS, c = (e * V) % COLS;
            float f[V];
            unpack16(buf[u], src, f);
            const float sc = scale ? scale[k] : 1.f;
#pragma unroll
            for (int v = 0; v < V; ++v) dst[k * ds + c + v] = sc * f[v];
        }
    }
}

// C B^T of one chunk and B/C group into cbg: Q x Q (both triangles; the heads take j <= i),
// one CTA, 4 x 4 tiles, the products' odd-stride shared-memory layout.
template <int RM, int CN> __device__ __forceinline__ void zero(float (&acc)[RM][CN]);
template <int RM, int CN>
__device__ __forceinline__ void mm(float (&acc)[RM][CN], const float *A, int am, int ak, const float *Bm, int bk,
                                   int bn, int K, int tm, int tn);
template <typename IO, int N, int P>
__global__ void __launch_bounds__(kCT) bwd_chunk_cb(BwdCParams p) {
    constexpr int Q = chunk_len<N, P>(), NS = N + 1, RM = Q / 16, CQ = Q / 16;
    extern __shared__ float sm[];
    float *sB = sm, *sC = sm + Q * NS;
    const int c = blockIdx.x, g = blockIdx.y, bi = blockIdx.z, tid = threadIdx.x;
    const int64_t t0 = (int64_t)c * Q;
    const int L = (int)min((int64_t)Q, (int64_t)p.T - t0);
    const int64_t tok0 = (int64_t)bi * p.T + t0;
    load_tile<IO, Q, N>(sB, NS, static_cast<const IO *>(p.B), tok0 * p.G * N + (int64_t)g * N, (int64_t)p.G * N, L);
    load_tile<IO, Q, N>(sC, NS, static_cast<const IO *>(p.C), tok0 * p.G * N + (int64_t)g * N, (int64_t)p.G * N, L);
    __syncthreads();
    const int tm = tid >> 4, tn = tid & 15;
    float acb[RM][CQ];
    zero(acb);
    mm(acb, sC, NS, 1, sB, 1, NS, N, tm, tn);
    float *out = p.cbg + (((int64_t)bi * p.nc + c) * p.G + g) * Q * Q;
#pragma unroll
    for (int a = 0; a < RM; ++a)
#pragma unroll
        for (int j = 0; j < CQ; ++j) out[(tm + 16 * a) * Q + tn + 16 * j] = acb[a][j];
}

// One chunk and head: its state s = B^T (w o X) into states and r = C^T (e o dY) into gst,
// and the sum of dt A over it into csum.  Both N x P products in the 2-D tiles of mm (thread
// (tm, tn): state rows tm + 16 a, columns tn + 16 j), whose loads are one wavefront each.  Two
// CTAs per SM (99 KB of shared memory each at N 128; registers capped at 128 for it).
template <typename IO, int N, int P>
__global__ void __launch_bounds__(kCT, N * P > 8192 ? 1 : 2) bwd_chunk_sr(BwdCParams p) {
    constexpr int Q = chunk_len<N, P>();
    extern __shared__ float sm[];
    float *sCe = sm;                  // [Q][N] e o C
    float *sBw = sCe + Q * N;         // [Q][N] w o B
    float *sdY = sBw + Q * N;         // [Q][P]
    float *sX = sdY + Q * P;          // [Q][P]
    float *cum = sX + Q * P;          // [Q]
    float *ev = cum + Q, *wv = ev + Q;
    const int c = blockIdx.x, h = blockIdx.y, bi = blockIdx.z, tid = threadIdx.x;
    const int64_t t0 = (int64_t)c * Q;
    const int L = (int)min((int64_t)Q, (int64_t)p.T - t0);
    const int g = h / (p.H / p.G);
    const int64_t tok0 = (int64_t)bi * p.T + t0;
    const int64_t bh = (int64_t)bi * p.H + h;
    load_tile<IO, Q, P>(sdY, P, static_cast<const IO *>(p.dy), tok0 * p.H * P + (int64_t)h * P, (int64_t)p.H * P, L);
    load_tile<IO, Q, P>(sX, P, static_cast<const IO *>(p.x), tok0 * p.H * P + (int64_t)h * P, (int64_t)p.H * P, L);
    chunk_cum<Q>(p.dt + tok0 * p.H + h, p.H, p.A[h], L, cum);
    if (tid < Q) {
        ev[tid] = expf(cum[tid]);
        wv[tid] = expf(cum[Q - 1] - cum[tid]);
    }
    if (tid == 0) p.csum[bh * p.nc + c] = cum[Q - 1];
    __syncthreads();
    load_tile<IO, Q, N>(sCe, N, static_cast<const IO *>(p.C), tok0 * p.G * N + (int64_t)g * N, (int64_t)p.G * N, L, ev);
    load_tile<IO, Q, N>(sBw, N, static_cast<const IO *>(p.B), tok0 * p.G * N + (int64_t)g * N, (int64_t)p.G * N, L, wv);
    __syncthreads();
    constexpr int RN = N / 16, CP = P / 16;
    const int tm = tid >> 4, tn = tid & 15;
    float ar[RN][CP], as[RN][CP];
    zero(ar);
    zero(as);
    mm(ar, sCe, 1, N, sdY, P, 1, Q, tm, tn);      // A(n, k) = (e o C)[k][n], Bop(k, q) = dY[k][q]
    mm(as, sBw, 1, N, sX, P, 1, Q, tm, tn);       // A(n, k) = (w o B)[k][n], Bop(k, q) = X[k][q]
    float *outr = p.gst + (bh * p.nc + c) * N * P;
    float *outs = p.states + (bh * p.nc + c) * N * P;
#pragma unroll
    for (int a = 0; a < RN; ++a)
#pragma unroll
        for (int j = 0; j < CP; ++j) {
            const int64_t o = (int64_t)(tm + 16 * a) * P + tn + 16 * j;
            outr[o] = ar[a][j];
            outs[o] = as[a][j];
        }
}

// The adjoint chain over chunks, backwards, per (batch row, head, state entry): g starts at
// dfinal; chunk c's slot receives g (the adjoint at the chunk's end) in place of its r, and
// g becomes e^{sum of dt A over chunk c} g + r.  What is left at the front is dinit.
constexpr int kRevU = 16;
__global__ void __launch_bounds__(kCT) bwd_state_reverse(BwdCParams p) {
    const int h = blockIdx.y, bi = blockIdx.z;
    const int64_t NP = (int64_t)p.N * p.P;
    const int64_t o = (int64_t)blockIdx.x * kCT + threadIdx.x;
    if (o >= NP) return;
    const int64_t bh = (int64_t)bi * p.H + h;
    float g = p.dfinal ? p.dfinal[bh * NP + o] : 0.f;
    float *gs = p.gst + bh * p.nc * NP + o;
    const float *cs = p.csum + bh * p.nc;
    int c = p.nc - 1;
    for (; c + 1 >= kRevU; c -= kRevU) {
        float rv[kRevU], cv[kRevU];
#pragma unroll
        for (int u = 0; u < kRevU; ++u) {
            rv[u] = gs[(int64_t)(c - u) * NP];
            cv[u] = cs[c - u];
        }
#pragma unroll
        for (int u = 0; u < kRevU; ++u) {
            gs[(int64_t)(c - u) * NP] = g;
            g = fmaf(expf(cv[u]), g, rv[u]);
        }
    }
    for (; c >= 0; --c) {
        const float r = gs[(int64_t)c * NP];
        gs[(int64_t)c * NP] = g;
        g = fmaf(expf(cs[c]), g, r);
    }
    if (p.dinit) p.dinit[bh * NP + o] = g;
}

// acc[a][j] += sum_k A(m_a, k) Bop(k, n_j) over this thread's outputs m_a = tm + 16 a,
// n_j = tn + 16 j, with A(m, k) = A[m * am + k * ak] and Bop(k, n) = Bm[k * bk + n * bn].
// Thread (tm, tn) = (tid / 16, tid % 16): a half warp shares its rows (broadcast loads of A),
// and its 16 lanes read 16 consecutive columns, or columns an odd stride apart, of Bop
// (distinct banks: every shared array below has an odd row stride).
template <int RM, int CN>
__device__ __forceinline__ void mm(float (&acc)[RM][CN], const float *A, int am, int ak, const float *Bm, int bk,
                                   int bn, int K, int tm, int tn) {
#pragma unroll 8
    for (int k = 0; k < K; ++k) {
        float av[RM], bv[CN];
#pragma unroll
        for (int a = 0; a < RM; ++a) av[a] = A[(tm + 16 * a) * am + k * ak];
#pragma unroll
        for (int j = 0; j < CN; ++j) bv[j] = Bm[k * bk + (tn + 16 * j) * bn];
#pragma unroll
        for (int a = 0; a < RM; ++a)
#pragma unroll
            for (int j = 0; j < CN; ++j) acc[a][j] = fmaf(av[a], bv[j], acc[a][j]);
    }
}

// The same product where the contraction runs over a triangle of a Q x Q factor (Q = 16 RM):
// output row m_a = tm + 16 a takes k in the 16-wide blocks s <= a (LOWER: A(m, k) = 0 for
// k > m's block) or s >= a (upper).  Row a's block is a for every thread, so every thread
// skips the same segments; inside the row's own block the zeros of the triangle are
// multiplied as they are.
template <int RM, int CN, bool LOWER>
__device__ __forceinline__ void mm_tri(float (&acc)[RM][CN], const float *A, int am, int ak, const float *Bm, int bk,
                                       int bn, int tm, int tn) {
#pragma unroll
    for (int sg = 0; sg < RM; ++sg) {
#pragma unroll 8
        for (int k = 16 * sg; k < 16 * sg + 16; ++k) {
            float av[RM], bv[CN];
#pragma unroll
            for (int a = 0; a < RM; ++a)
                if (LOWER ? a >= sg : a <= sg) av[a] = A[(tm + 16 * a) * am + k * ak];
#pragma unroll
            for (int j = 0; j < CN; ++j) bv[j] = Bm[k * bk + (tn + 16 * j) * bn];
#pragma unroll
            for (int a = 0; a < RM; ++a)
                if (LOWER ? a >= sg : a <= sg) {
#pragma unroll
                    for (int j = 0; j < CN; ++j) acc[a][j] = fmaf(av[a], bv[j], acc[a][j]);
                }
        }
    }
}

// The product on the lower block triangle of a Q x Q output (column blocks j <= row block a).
template <int RM, int CN>
__device__ __forceinline__ void mm_lowout(float (&acc)[RM][CN], const float *A, int am, int ak, const float *Bm,
                                          int bk, int bn, int K, int tm, int tn) {
#pragma unroll 8
    for (int k = 0; k < K; ++k) {
        float av[RM], bv[CN];
#pragma unroll
        for (int a = 0; a < RM; ++a) av[a] = A[(tm + 16 * a) * am + k * ak];
#pragma unroll
        for (int j = 0; j < CN; ++j) bv[j] = Bm[k * bk + (tn + 16 * j) * bn];
#pragma unroll
        for (int a = 0; a < RM; ++a)
#pragma unroll
            for (int j = 0; j < CN; ++j)
                if (j <= a) acc[a][j] = fmaf(av[a], bv[j], acc[a][j]);
    }
}

template <int RM, int CN> __device__ __forceinline__ void zero(float (&acc)[RM][CN]) {
#pragma unroll
    for (int a = 0; a < RM; ++a)
#pragma unroll
        for (int j = 0; j < CN; ++j) acc[a][j] = 0.f;
}

// sum over the 16 lanes of a half warp
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int N, int P>
constexpr size_t chunk_grad_floats() {
    return grad_floats(N, P, chunk_len<N, P>());
}

template <typename IO, int N, int P>
__global__ void __launch_bounds__(kCT, 1) bwd_chunk_grad(BwdCParams p) {
    constexpr int Q = chunk_len<N, P>(), QS = Q + 1, PS = P + 1, NS = N + 1;
    constexpr int RM = Q / 16, CQ = Q / 16, CP = P / 16, CN = N / 16;
    extern __shared__ float sm[];
    double *redd = reinterpret_cast<double *>(sm);   // [2]: <g, h>, dA (8-byte aligned at the start)
    float *red = sm + 4;              // [2]: dD
    float *sX = sm + 8;               // [Q][PS]   x
    float *sdY = sX + Q * PS;         // [Q][PS]   dy
    float *sB = sdY + Q * PS;         // [Q][NS]   B
    float *sC = sB + Q * NS;          // [Q][NS]   C
    float *sH = sC + Q * NS;          // [N][PS]   state entering the chunk
    float *sGc = sH + N * PS;         // [N][PS]   adjoint at the chunk's end
    float *sS = sGc + N * PS;         // [Q][QS]   S
    float *sG = sS + Q * QS;          // [Q][QS]   G
    float *sK = sG + Q * QS;          // [Q][QS]   K, then its row prefix sums
    float *cum = sK + Q * QS;         // [Q]
    float *wv = cum + Q, *ev = wv + Q;
    float *wvv = ev + Q, *eu = wvv + Q;   // [Q] w_j v_j, e_i u_i
    const int c = blockIdx.x, h = blockIdx.y, bi = blockIdx.z, tid = threadIdx.x;
    const int tm = tid >> 4, tn = tid & 15;
    const int64_t t0 = (int64_t)c * Q;
    const int L = (int)min((int64_t)Q, (int64_t)p.T - t0);
    const int g = h / (p.H / p.G);
    const int64_t bh = (int64_t)bi * p.H + h;
    const int64_t tok0 = (int64_t)bi * p.T + t0;
    const float Ah = p.A[h];

    load_tile<IO, Q, P>(sX, PS, static_cast<const IO *>(p.x), tok0 * p.H * P + (int64_t)h * P, (int64_t)p.H * P, L);
    load_tile<IO, Q, P>(sdY, PS, static_cast<const IO *>(p.dy), tok0 * p.H * P + (int64_t)h * P, (int64_t)p.H * P, L);
    load_tile<IO, Q, N>(sB, NS, static_cast<const IO *>(p.B), tok0 * p.G * N + (int64_t)g * N, (int64_t)p.G * N, L);
    load_tile<IO, Q, N>(sC, NS, static_cast<const IO *>(p.C), tok0 * p.G * N + (int64_t)g * N, (int64_t)p.G * N, L);
    load_tile<float, N, P>(sH, PS, p.states, (bh * p.nc + c) * N * P, P, N);
    load_tile<float, N, P>(sGc, PS, p.gst, (bh * p.nc + c) * N * P, P, N);
    if (tid < 2) {
        redd[tid] = 0.0;
        red[tid] = 0.f;
    }
    chunk_cum<Q>(p.dt + tok0 * p.H + h, p.H, Ah, L, cum);
    if (tid < Q) {
        wv[tid] = expf(cum[Q - 1] - cum[tid]);
        ev[tid] = expf(cum[tid]);
    }
    __syncthreads();

    // C B^T (formed once per group) and dY X^T; S, G and K = G o (C B^T)
    {
        float acb[RM][CQ], ayx[RM][CQ];
        {
            const float *cb = p.cbg + (((int64_t)bi * p.nc + c) * p.G + g) * Q * Q;
#pragma unroll
            for (int a = 0; a < RM; ++a)
#pragma unroll
                for (int j = 0; j < CQ; ++j) acb[a][j] = __ldg(cb + (tm + 16 * a) * Q + tn + 16 * j);
        }
        zero(ayx);
        mm_lowout(ayx, sdY, PS, 1, sX, 1, PS, P, tm, tn);        // only j <= i is used
#pragma unroll
        for (int a = 0; a < RM; ++a) {
            const int i = tm + 16 * a;
#pragma unroll
            for (int j = 0; j < CQ; ++j) {
                const int jj = tn + 16 * j;
                float sv = 0.f, gv = 0.f;
                if (jj <= i) {
                    const float l = expf(cum[i] - cum[jj]);
                    sv = l * acb[a][j];
                    gv = l * ayx[a][j];
                }
                sS[i * QS + jj] = sv;
                sG[i * QS + jj] = gv;
                sK[i * QS + jj] = gv * acb[a][j];
            }
        }
    }
    __syncthreads();

    // dX = S^T dY + w o (B g) + D dY;  v_j = x_j.(B g)_j;  dD
    {
        float asd[RM][CP], abg[RM][CP];
        zero(asd);
        zero(abg);
        mm_tri<RM, CP, false>(asd, sS, 1, QS, sdY, PS, 1, tm, tn);   // sum over i >= j
        mm(abg, sB, NS, 1, sGc, PS, 1, N, tm, tn);
        const float Dh = p.D ? p.D[h] : 0.f;
        IO *dx = static_cast<IO *>(p.dx);
        float dd = 0.f;
#pragma unroll
        for (int a = 0; a < RM; ++a) {
            const int j = tm + 16 * a;
            float vj = 0.f;
#pragma unroll
            for (int k = 0; k < CP; ++k) {
                const int q = tn + 16 * k;
                const float xv = sX[j * PS + q], dyv = sdY[j * PS + q];
                vj = fmaf(abg[a][k], xv, vj);
                dd = fmaf(dyv, xv, dd);
                if (j < L) stf(dx, (tok0 + j) * p.H * P + (int64_t)h * P + q, fmaf(wv[j], abg[a][k], fmaf(Dh, dyv, asd[a][k])));
            }
            vj = sum16(vj);
            if (tn == 0) wvv[j] = wv[j] * vj;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
        if ((tid & 31) == 0) atomicAdd(red + 0, dd);
    }

    // dC = G B + e o (dY h^T);  u_i = C_i.(h dY_i)
    {
        float agb[RM][CN], ayh[RM][CN];
        zero(agb);
        zero(ayh);
        mm_tri<RM, CN, true>(agb, sG, QS, 1, sB, NS, 1, tm, tn);    // sum over j <= i
        mm(ayh, sdY, PS, 1, sH, 1, PS, P, tm, tn);
#pragma unroll
        for (int a = 0; a < RM; ++a) {
            const int i = tm + 16 * a;
            float ui = 0.f;
#pragma unroll
            for (int k = 0; k < CN; ++k) {
                const int n = tn + 16 * k;
                ui = fmaf(sC[i * NS + n], ayh[a][k], ui);
                if (i < L) p.dCh[((tok0 + i) * p.H + h) * N + n] = fmaf(ev[i], ayh[a][k], agb[a][k]);
            }
            ui = sum16(ui);
            if (tn == 0) eu[i] = ev[i] * ui;
        }
    }

    // dB = G^T C + w o (X g^T)
    {
        float agc[RM][CN], axg[RM][CN];
        zero(agc);
        zero(axg);
        mm_tri<RM, CN, false>(agc, sG, 1, QS, sC, NS, 1, tm, tn);   // sum over i >= j
        mm(axg, sX, PS, 1, sGc, 1, PS, P, tm, tn);
#pragma unroll
        for (int a = 0; a < RM; ++a) {
            const int j = tm + 16 * a;
            if (j < L) {
#pragma unroll
                for (int k = 0; k < CN; ++k)
                    p.dBh[((tok0 + j) * p.H + h) * N + tn + 16 * k] = fmaf(wv[j], axg[a][k], agc[a][k]);
            }
        }
    }

    // <g, h> (fp32 per thread, double across threads); row prefix sums of K (exclusive)
    {
        float gh = 0.f;
        for (int e = tid; e < N * P; e += kCT) {
            const int n = e / P, q = e % P;
            gh = fmaf(sGc[n * PS + q], sH[n * PS + q], gh);
        }
        double ghd = gh;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ghd += __shfl_xor_sync(0xffffffffu, ghd, o);
        if ((tid & 31) == 0) atomicAdd(redd + 0, ghd);
        // exclusive prefix sums along each row of K: TPR threads per row, Q / TPR entries each
        constexpr int TPR = kCT / Q, EPT = Q / TPR;
        static_assert(TPR * Q == kCT && TPR <= 32, "whole rows of K per warp");
        const int i = tid / TPR, part = tid % TPR;
        float loc[EPT];
        float run = 0.f;
#pragma unroll
        for (int jj = 0; jj < EPT; ++jj) {
            loc[jj] = run;
            run += sK[i * QS + part * EPT + jj];
        }
        float v = run;
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o, TPR);
            if (part >= o) v += u;
        }
        const float off = v - run;
#pragma unroll
        for (int jj = 0; jj < EPT; ++jj) sK[i * QS + part * EPT + jj] = loc[jj] + off;
    }
    __syncthreads();

    // rc_k, TPR threads per token (fp32 partial sums, combined in double); ddt, dA and dD
    {
        constexpr int TPR = kCT / Q;
        const int k = tid / TPR, part = tid % TPR;
        float cs = 0.f, es = 0.f, ws = 0.f;
        for (int ii = part; ii < Q; ii += TPR) {
            if (ii >= k) {
                cs += sK[ii * QS + k];
                es += eu[ii];
            } else {
                ws += wvv[ii];
            }
        }
        double rc = (double)cs + (double)es + (double)ws;
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) rc += __shfl_xor_sync(0xffffffffu, rc, o);
        rc += exp((double)cum[Q - 1]) * redd[0];
        double da = 0.0;
        if (part == 0 && k < L) {
            const int64_t o = (tok0 + k) * p.H + h;
            p.ddt[o] = (float)(Ah * rc);
            da = (double)p.dt[o] * rc;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
        if ((tid & 31) == 0) atomicAdd(redd + 1, da);
    }
    __syncthreads();
    if (tid == 0) {
        atomicAdd(p.dA + h, (float)redd[1]);
        if (p.dD) atomicAdd(p.dD + h, red[0]);
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

// ---- chunked path: host side ----
int chunk_q(const Problem &p) { return chunk_len_of((int)p.N, (int)p.P); }

// the chunked path's domain: scalar A at the head dims its kernels are built for
bool chunked_applies(const Problem &p) {
    if (p.a_mode != SSD_A_SCALAR || (p.P != 64 && p.P != 128)) return false;
    if (p.N != 64 && p.N != 128 && p.N != 256) return false;
    const int Q = chunk_q(p);
    if (Q == 0) return false;
    if (p.H > 65535 || p.b > 65535 || (p.T + Q - 1) / Q > (int64_t)INT32_MAX) return false;
    Problem q = p;
    q.Q = Q;
    q.nc = (p.T + Q - 1) / Q;
    return generic_supports(q);
}

struct BwdCLayout {
    int64_t nc;
    size_t off_cs, off_st, off_g, off_dbh, off_dch, off_cb, total;
};

BwdCLayout bwdc_layout(const Problem &p) {
    BwdCLayout l;
    const int Q = chunk_q(p);
    l.nc = (p.T + Q - 1) / Q;
    const size_t tokh = (size_t)(p.b * p.T * p.H), np = (size_t)(p.b * p.H * l.nc * p.N * p.P);
    l.off_cs = kStatusBytes;
    l.off_st = align_up(l.off_cs + sizeof(float) * (size_t)(p.b * p.H * l.nc), 256);
    l.off_g = align_up(l.off_st + sizeof(float) * np, 256);
    l.off_dbh = align_up(l.off_g + sizeof(float) * np, 256);
    l.off_dch = align_up(l.off_dbh + sizeof(float) * tokh * p.N, 256);
    l.off_cb = align_up(l.off_dch + sizeof(float) * tokh * p.N, 256);
    l.total = align_up(l.off_cb + sizeof(float) * (size_t)(p.b * l.nc * p.G) * Q * Q, 256);
    return l;
}

template <typename IO, int N, int P>
cudaError_t launch_chunked_typed(const Problem &p, const BwdCParams &cp, cudaStream_t s) {
    constexpr int Q = chunk_len<N, P>();
    static_assert(Q > 0, "an instantiated head shape has a chunk length");
    const size_t sm_r = sizeof(float) * (size_t)(2 * Q * N + 2 * Q * P + 3 * Q);
    const size_t sm_g = sizeof(float) * chunk_grad_floats<N, P>();
    cudaError_t e = cudaFuncSetAttribute(bwd_chunk_sr<IO, N, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_r);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_chunk_grad<IO, N, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_g);
    if (e != cudaSuccess) return e;
    const size_t sm_cb = sizeof(float) * (size_t)(2 * Q * (N + 1));
    if ((e = cudaFuncSetAttribute(bwd_chunk_cb<IO, N, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_cb)) !=
        cudaSuccess)
        return e;
    bwd_chunk_cb<IO, N, P><<<dim3((unsigned)cp.nc, (unsigned)p.G, (unsigned)p.b), kCT, sm_cb, s>>>(cp);
    const dim3 grid((unsigned)cp.nc, (unsigned)p.H, (unsigned)p.b);
    bwd_chunk_sr<IO, N, P><<<grid, kCT, sm_r, s>>>(cp);
    // the state entering every chunk: the generic forward's state passing, in place
    {
        Problem q = p;
        q.Q = Q;
        q.nc = cp.nc;
        q.y = nullptr;
        q.final_state = nullptr;
        GenericWorkspace gw;
        gw.status = nullptr;
        gw.chunk_sum = cp.csum;
        gw.states = cp.states;
        if ((e = generic_passing_launch(q, gw, s)) != cudaSuccess) return e;
    }
    bwd_state_reverse<<<dim3((unsigned)((N * P + kCT - 1) / kCT), (unsigned)p.H, (unsigned)p.b), kCT, 0, s>>>(cp);
    record_dominant_start(s);
    bwd_chunk_grad<IO, N, P><<<grid, kCT, sm_g, s>>>(cp);
    record_dominant_stop(s);
    note_launches(4);
    return cudaGetLastError();
}

cudaError_t chunked_launch(const Problem &p, const BwdGrads &gr, char *base, cudaStream_t s) {
    const BwdCLayout l = bwdc_layout(p);
    cudaError_t e;
    BwdCParams cp;
    cp.x = p.x; cp.B = p.B; cp.C = p.C; cp.dy = gr.dy;
    cp.dt = p.dt; cp.A = p.A; cp.D = p.D; cp.dfinal = gr.dfinal;
    cp.dx = gr.dx; cp.ddt = gr.ddt; cp.dA = gr.dA; cp.dD = gr.dD; cp.dinit = gr.dinit;
    cp.states = reinterpret_cast<float *>(base + l.off_st);
    cp.csum = reinterpret_cast<float *>(base + l.off_cs);
    cp.gst = reinterpret_cast<float *>(base + l.off_g);
    cp.dBh = reinterpret_cast<float *>(base + l.off_dbh);
    cp.dCh = reinterpret_cast<float *>(base + l.off_dch);
    cp.cbg = reinterpret_cast<float *>(base + l.off_cb);
    cp.b = (int)p.b; cp.T = (int)p.T; cp.H = (int)p.H; cp.G = (int)p.G; cp.N = (int)p.N; cp.P = (int)p.P;
    cp.nc = (int)l.nc;
    const bool bf = p.io_dtype == SSD_DTYPE_BF16;
#define SSD_CHUNKED(N_, P_) \
    (bf ? launch_chunked_typed<__nv_bfloat16, N_, P_>(p, cp, s) : launch_chunked_typed<float, N_, P_>(p, cp, s))
    if (p.P == 64) e = p.N == 64 ? SSD_CHUNKED(64, 64) : p.N == 128 ? SSD_CHUNKED(128, 64) : SSD_CHUNKED(256, 64);
    else e = p.N == 64 ? SSD_CHUNKED(64, 128) : SSD_CHUNKED(128, 128);
#undef SSD_CHUNKED
    if (e != cudaSuccess) return e;
    // dB, dC: the per-head sums over each group's heads
    BwdParams bp;
    std::memset(&bp, 0, sizeof(bp));
    bp.dB = gr.dB; bp.dC = gr.dC;
    bp.dBh = cp.dBh; bp.dCh = cp.dCh;
    bp.b = (int)p.b; bp.T = (int)p.T; bp.H = (int)p.H; bp.N = (int)p.N; bp.G = (int)p.G;
    if (bf) bwd_finish_bc<__nv_bfloat16><<<1184, 256, 0, s>>>(bp);
    else bwd_finish_bc<float><<<1184, 256, 0, s>>>(bp);
    note_launches(1);
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

size_t bwd_workspace_bytes(const Problem &p, bool chunked_ok) {
    return chunked_ok && chunked_applies(p) ? bwdc_layout(p).total : bwd_layout(p).total;
}

cudaError_t bwd_launch(const Problem &p, const BwdGrads &gr, void *ws, cudaStream_t s, bool chunked_ok) {
    char *base = static_cast<char *>(ws);
    if (chunked_ok && chunked_applies(p)) {
        cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(gr.dA, 0, sizeof(float) * (size_t)p.H, s);
        if (e == cudaSuccess && gr.dD) e = cudaMemsetAsync(gr.dD, 0, sizeof(float) * (size_t)p.H, s);
        if (e != cudaSuccess) return e;
        return chunked_launch(p, gr, base, s);
    }
    const BwdLayout l = bwd_layout(p);
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
