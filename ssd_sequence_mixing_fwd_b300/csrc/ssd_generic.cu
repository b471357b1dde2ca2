// ssd_generic.cu -- the generic CUDA-core path of the SSD chunked scan.
//
// Three kernels, all arithmetic in fp32 (exact fp32 FMA, no tensor cores), for
// any dims the ABI accepts.  It is the path for fp32 inputs (where the 1e-5
// tolerance rules out tf32 operands) and for shapes the fused tcgen05 kernel
// does not take.  The steps are those of Structured State Space Duality, "The
// chunked algorithm takes both":
//
//   gen_chunk_state    per (b, h, chunk): the chunk prefix sums of the log
//                      decay, and the chunk's input projection
//                      s_c = B_c^T (w o X_c), w_j = decay from token j to the
//                      chunk end (the low-rank factor of the off-diagonal
//                      blocks).
//   gen_state_passing  per (b, h, n, p): h_c = a_c h_{c-1} + s_c over chunks,
//                      one recurrence step per chunk, fp32 ("When it breaks");
//                      leaves h_{c-1} (the state entering chunk c) in place.
//   gen_chunk_output   per (b, h, chunk, 32-row tile): the diagonal block
//                      (C B^T o L) X with L_ij = exp(cum_i - cum_j), plus the
//                      off-diagonal part exp(cum_i) C_i^T h_{c-1}, plus D x.
//
// In the diagonal-A variant the decay of state dim n between tokens j <= i is
// exp(A_{h,n} (S_i - S_j)) with S the chunk prefix sum of dt, so the mask is a
// sum over n.  In both variants the output kernel splits each tile's decay into
// a row and a column factor, so that the (i, j) products are plain dot products.
#include <cuda_bf16.h>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTT = 16;        // tokens per shared-memory tile (chunk state)
constexpr int kMaxAcc = 64;    // N*P / 256 accumulators per thread at most (chunk state)
constexpr int kPassU = 16;     // chunks whose states are loaded together (state passing)
constexpr int kRT = 32;        // output rows per block
constexpr int kJT = 32;        // key (j) columns per tile
constexpr int kMaxOut = 32;    // kRT*P / 256 outputs per thread at most

template <typename IO> __device__ __forceinline__ float ld_io(const IO *p, int64_t i);
template <> __device__ __forceinline__ float ld_io<float>(const float *p, int64_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
template <typename IO> __device__ __forceinline__ void st_io(IO *p, int64_t i, float v);
template <> __device__ __forceinline__ void st_io<float>(float *p, int64_t i, float v) { p[i] = v; }
template <> __device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

// dst[k * ds + c] = src[base + k * rs + c] for k < rows, c < cols (0 for k >= valid), as
// 16-byte loads when base, rs and cols allow it (8 bf16 or 4 fp32 per load; the pointers
// of the ABI are 16-byte aligned), else element by element.  All threads of the block.
template <typename IO>
__device__ __forceinline__ void load_tile(float *dst, int ds, const IO *src, int64_t base, int64_t rs, int rows,
                                          int valid, int cols) {
    constexpr int V = 16 / (int)sizeof(IO);
    if ((cols % V) == 0 && (base % V) == 0 && (rs % V) == 0) {
        const int cv = cols / V;
        for (int e = threadIdx.x; e < rows * cv; e += blockDim.x) {
            const int k = e / cv, c = (e % cv) * V;
            float *d = dst + k * ds + c;
            if (k < valid) {
                const uint4 u = *reinterpret_cast<const uint4 *>(src + base + k * rs + c);
                if constexpr (sizeof(IO) == 2) {
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        d[2 * q] = __uint_as_float(w[q] << 16);
                        d[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
                    }
                } else {
                    d[0] = __uint_as_float(u.x);
                    d[1] = __uint_as_float(u.y);
                    d[2] = __uint_as_float(u.z);
                    d[3] = __uint_as_float(u.w);
                }
            } else {
#pragma unroll
                for (int q = 0; q < V; ++q) d[q] = 0.f;
            }
        }
    } else {
        for (int e = threadIdx.x; e < rows * cols; e += blockDim.x) {
            const int k = e / cols, c = e % cols;
            dst[k * ds + c] = (k < valid) ? ld_io(src, base + k * rs + c) : 0.f;
        }
    }
}

// e^x for the decay factors.  fp32 io keeps expf (the fp32 tolerance is 1e-5);
// bf16 io (tolerance 2e-3) takes the hardware base-2 exponential, whose relative
// error is ~2^-22 -- the inner loop of the diagonal-A output kernel evaluates one
// decay per (i, j, n), and expf's range reduction made it the bulk of the time.
template <typename IO> __device__ __forceinline__ float dexp(float x);
template <> __device__ __forceinline__ float dexp<float>(float x) { return expf(x); }
template <> __device__ __forceinline__ float dexp<__nv_bfloat16>(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

// Inclusive prefix sum over the chunk of s_t = dt_t*A_h (scalar) or dt_t
// (diagonal) into lcum[0..Q); entries past the chunk's length are zero.
// Hillis-Steele over shared memory; Q <= blockDim.
__device__ __forceinline__ void chunk_prefix(const Problem &p, int bi, int h, int64_t t0, int L,
                                             float *lcum) {
    const int tid = threadIdx.x;
    float v = 0.f;
    if (tid < L) {
        v = p.dt[((int64_t)bi * p.T + t0 + tid) * p.H + h];
        if (p.a_mode == SSD_A_SCALAR) v *= p.A[h];
    }
    if (tid < p.Q) lcum[tid] = v;
    __syncthreads();
    for (int off = 1; off < p.Q; off <<= 1) {
        float add = (tid < p.Q && tid >= off) ? lcum[tid - off] : 0.f;
        __syncthreads();
        if (tid < p.Q) lcum[tid] += add;
        __syncthreads();
    }
}

template <typename IO, int ACC>
__global__ void __launch_bounds__(kThreads) gen_chunk_state(Problem p, GenericWorkspace w) {
    extern __shared__ float smem[];
    const int c = blockIdx.x, h = blockIdx.y, bi = blockIdx.z, tid = threadIdx.x;
    const int N = (int)p.N, P = (int)p.P;
    const int64_t t0 = (int64_t)c * p.Q;
    const int L = (int)min(p.Q, p.T - t0);
    const int g = h / (int)(p.H / p.G);
    const IO *X = static_cast<const IO *>(p.x);
    const IO *Bm = static_cast<const IO *>(p.B);

    const int NW = (N + 3) & ~3;        // Bw row stride (float4 rows)
    float *lcum = smem;                 // Q
    float *Bw = smem + ((p.Q + 3) & ~3);   // kTT x NW, 16-byte aligned rows
    float *Xs = Bw + kTT * NW;          // kTT x P

    chunk_prefix(p, bi, h, t0, L, lcum);
    const float total = lcum[L - 1];
    if (tid == 0) w.chunk_sum[((int64_t)bi * p.H + h) * p.nc + c] = total;

    // thread: column pcol of the state and the ACC consecutive state rows from nbase
    // (ACC >= N / (threads / P), a power of two), read from Bw as float4
    const int pcol = tid % P;
    const int nbase = (tid / P) * ACC;
    float acc[ACC];
#pragma unroll
    for (int a = 0; a < ACC; ++a) acc[a] = 0.f;

    for (int tt = 0; tt < L; tt += kTT) {
        for (int e = tid; e < kTT * N; e += kThreads) {
            const int k = e / N, n = e % N;
            float v = 0.f;
            if (tt + k < L) {
                const int64_t tok = (int64_t)bi * p.T + t0 + tt + k;
                const float d = total - lcum[tt + k];
                const float lw = (p.a_mode == SSD_A_SCALAR) ? d : p.A[(int64_t)h * N + n] * d;
                v = ld_io(Bm, (tok * p.G + g) * N + n) * dexp<IO>(lw);
            }
            Bw[k * NW + n] = v;
        }
        load_tile(Xs, P, X, (((int64_t)bi * p.T + t0 + tt) * p.H + h) * P, (int64_t)p.H * P, kTT, L - tt, P);
        __syncthreads();
        if (nbase < N) {
#pragma unroll 4
            for (int k = 0; k < kTT; ++k) {
                const float xv = Xs[k * P + pcol];
                const float *bk = Bw + k * NW + nbase;
#pragma unroll
                for (int a = 0; a < ACC; a += 4) {
                    if (nbase + a < NW) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(bk + a);
                        acc[a] = fmaf(b4.x, xv, acc[a]);
                        acc[a + 1] = fmaf(b4.y, xv, acc[a + 1]);
                        acc[a + 2] = fmaf(b4.z, xv, acc[a + 2]);
                        acc[a + 3] = fmaf(b4.w, xv, acc[a + 3]);
                    }
                }
            }
        }
        __syncthreads();
    }
    float *out = w.states + (((int64_t)bi * p.H + h) * p.nc + c) * N * P;
#pragma unroll
    for (int a = 0; a < ACC; ++a) {
        const int n = nbase + a;
        if (n < N) out[(int64_t)n * P + pcol] = acc[a];
    }
}

__global__ void __launch_bounds__(kThreads) gen_state_passing(Problem p, GenericWorkspace w) {
    const int h = blockIdx.y, bi = blockIdx.z;
    const int64_t NP = p.N * p.P;
    const int64_t o = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (o >= NP) return;
    const int n = (int)(o / p.P);
    const int64_t bh = (int64_t)bi * p.H + h;
    float hs = p.init ? p.init[bh * NP + o] : 0.f;
    float *st = w.states + bh * p.nc * NP + o;
    const float *cs = w.chunk_sum + bh * p.nc;
    const float An = (p.a_mode == SSD_A_SCALAR) ? 1.f : p.A[(int64_t)h * p.N + n];
    // the loads of kPassU chunks are issued together (the recurrence itself is a
    // chain of FMAs; one load in flight per thread left the kernel latency-bound)
    int64_t c = 0;
    for (; c + kPassU <= p.nc; c += kPassU) {
        float sv[kPassU], cv[kPassU];
#pragma unroll
        for (int u = 0; u < kPassU; ++u) {
            sv[u] = st[(c + u) * NP];
            cv[u] = cs[c + u];
        }
#pragma unroll
        for (int u = 0; u < kPassU; ++u) {
            st[(c + u) * NP] = hs;             // state entering chunk c + u
            hs = fmaf(expf(An * cv[u]), hs, sv[u]);   // decay across the whole chunk
        }
    }
    for (; c < p.nc; ++c) {
        const float s = st[c * NP];
        st[c * NP] = hs;
        hs = fmaf(expf(An * cs[c]), hs, s);
    }
    if (p.final_state) p.final_state[bh * NP + o] = hs;
}

template <typename IO>
__global__ void __launch_bounds__(kThreads) gen_chunk_output(Problem p, GenericWorkspace w) {
    extern __shared__ float smem[];
    const int nrt = (int)((p.Q + kRT - 1) / kRT);
    const int c = blockIdx.x / nrt, rt = blockIdx.x % nrt;
    const int h = blockIdx.y, bi = blockIdx.z, tid = threadIdx.x;
    const int N = (int)p.N, P = (int)p.P;
    const int64_t t0 = (int64_t)c * p.Q;
    const int L = (int)min(p.Q, p.T - t0);
    const int i0 = rt * kRT;
    if (i0 >= L) return;                       // uniform over the block
    const int g = h / (int)(p.H / p.G);
    const IO *X = static_cast<const IO *>(p.x);
    const IO *Bm = static_cast<const IO *>(p.B);
    const IO *Cm = static_cast<const IO *>(p.C);
    const int NS = N + 1;                      // padded row stride

    float *lcum = smem;                        // Q
    float *As = lcum + p.Q;                    // N
    float *Cs = As + N;                        // kRT x NS
    float *Bs = Cs + kRT * NS;                 // kJT x NS
    float *Xs = Bs + kJT * NS;                 // kJT x P
    // kJT x P tile of h_{c-1}: only after the column tiles, in the B and X tiles' space
    // (kJT * (NS + P) >= kJT * P floats)
    float *Hs = Bs;
    // transposed buffers, read as float4 (16-byte aligned): S of a tile (ST[k][r]) and a
    // decayed C (CT[n][r]: the row factor of a split diagonal-A tile, then e^{cum_i} C)
    float *ST = smem + ((Xs + kJT * P - smem + 3) & ~3);   // kJT x kRT
    float *CT = ST + kJT * kRT;                            // N x kRT

    chunk_prefix(p, bi, h, t0, L, lcum);
    for (int n = tid; n < N; n += kThreads)
        As[n] = (p.a_mode == SSD_A_SCALAR) ? 1.f : p.A[(int64_t)h * N + n];
    load_tile(Cs, NS, Cm, (((int64_t)bi * p.T + t0 + i0) * p.G + g) * N, (int64_t)p.G * N, kRT, L - i0, N);
    __syncthreads();
    // the largest |A_n| bounds the factors of the split decay below (scalar A: its cum
    // already carries A, and As = 1)
    float amax = 0.f;
    for (int n = 0; n < N; ++n) amax = fmaxf(amax, fabsf(As[n]));

    // Each thread owns column pcol of y and the nout consecutive rows from rbase, so that a
    // k step of a product reads one value of its column and the rows' values as float4.
    const int pcol = tid % P;
    const int rblocks = kThreads / P;          // >= 1 since P <= 256
    const int nout = rblocks >= kRT ? 1 : kRT / rblocks;
    const int rbase = (tid / P) * nout;
    const bool active = rbase < kRT;
    float acc[kMaxOut];
#pragma unroll
    for (int a = 0; a < kMaxOut; ++a) acc[a] = 0.f;
    // acc[a] += v[a] * x for the thread's rows, v = the nout values at vk (16-byte aligned)
    auto accumulate = [&](const float *vk, float x) {
        if (nout >= 4) {
#pragma unroll
            for (int a = 0; a < kMaxOut; a += 4) {
                if (a < nout) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(vk + a);
                    acc[a] = fmaf(v4.x, x, acc[a]);
                    acc[a + 1] = fmaf(v4.y, x, acc[a + 1]);
                    acc[a + 2] = fmaf(v4.z, x, acc[a + 2]);
                    acc[a + 3] = fmaf(v4.w, x, acc[a + 3]);
                }
            }
        } else {
#pragma unroll
            for (int a = 0; a < 4; ++a)
                if (a < nout) acc[a] = fmaf(vk[a], x, acc[a]);
        }
    };

    const int i_last = min(i0 + kRT, L) - 1;
    for (int j0 = 0; j0 <= i_last; j0 += kJT) {
        load_tile(Bs, NS, Bm, (((int64_t)bi * p.T + t0 + j0) * p.G + g) * N, (int64_t)p.G * N, kJT, L - j0, N);
        load_tile(Xs, P, X, (((int64_t)bi * p.T + t0 + j0) * p.H + h) * P, (int64_t)p.H * P, kJT, L - j0, P);
        __syncthreads();
        // e^{A_n (cum_i - cum_j)} = e^{A_n (cum_i - R)} e^{A_n (R - cum_j)} (scalar A: A_n = 1 and
        // cum carries A).  With the first factor folded into C (transposed, CT) and the second
        // into B, the tile is a plain dot product over n, computed four rows per thread (no
        // exponential inside).  R = cum at the column tile's last token when the tile lies left
        // of the rows (both factors <= 1); for the tile on the diagonal, R = cum at its middle
        // row, taken only while amax * (half the tile's cum range) keeps the factors inside
        // fp32 (< e^80); otherwise that tile is evaluated directly.
        const int jl = min(j0 + kJT, L) - 1;
        const bool below = jl < i0;
        const float Rt = below ? lcum[jl] : lcum[min(i0 + kRT / 2, L) - 1];
        const bool split = below || amax * fmaxf(fabsf(lcum[i_last] - Rt), fabsf(Rt - lcum[j0])) < 80.f;
        if (split) {
            for (int e = tid; e < N * kRT; e += kThreads) {
                const int n = e / kRT, r = e % kRT;
                const int i = i0 + r;
                CT[n * kRT + r] = (i < L) ? Cs[r * NS + n] * dexp<IO>(As[n] * (lcum[i] - Rt)) : 0.f;
            }
            for (int e = tid; e < kJT * N; e += kThreads) {
                const int k = e / N, n = e % N;
                const int j = j0 + k;
                Bs[k * NS + n] = (j < L) ? Bs[k * NS + n] * dexp<IO>(As[n] * (Rt - lcum[j])) : 0.f;
            }
            __syncthreads();
            static_assert(kRT == 32 && kJT == 32 && kThreads == 256, "4 rows x 1 column per thread");
            const int k = tid & 31, r4 = 4 * (tid >> 5);
            const float *br = Bs + k * NS;
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
            for (int n = 0; n < N; ++n) {
                const float4 c4 = *reinterpret_cast<const float4 *>(CT + n * kRT + r4);
                const float bv = br[n];
                d0 = fmaf(c4.x, bv, d0);
                d1 = fmaf(c4.y, bv, d1);
                d2 = fmaf(c4.z, bv, d2);
                d3 = fmaf(c4.w, bv, d3);
            }
            const int j = j0 + k, i = i0 + r4;
            *reinterpret_cast<float4 *>(ST + k * kRT + r4) =
                make_float4((j <= i && i < L) ? d0 : 0.f, (j <= i + 1 && i + 1 < L) ? d1 : 0.f,
                            (j <= i + 2 && i + 2 < L) ? d2 : 0.f, (j <= i + 3 && i + 3 < L) ? d3 : 0.f);
        } else {
            for (int e = tid; e < kRT * kJT; e += kThreads) {
                const int r = e % kRT, k = e / kRT;
                const int i = i0 + r, j = j0 + k;
                float v = 0.f;
                if (j <= i && i < L) {
                    const float dlt = lcum[i] - lcum[j];
                    const float *cr = Cs + r * NS;
                    const float *br = Bs + k * NS;
                    if (p.a_mode == SSD_A_SCALAR) {
                        float dot = 0.f;
                        for (int n = 0; n < N; ++n) dot = fmaf(cr[n], br[n], dot);
                        v = dot * dexp<IO>(dlt);
                    } else {
                        for (int n = 0; n < N; ++n) v = fmaf(cr[n] * br[n], dexp<IO>(As[n] * dlt), v);
                    }
                }
                ST[k * kRT + r] = v;
            }
        }
        __syncthreads();
        // Y_diag += S X (columns past the sequence end have X = 0)
        if (active)
            for (int k = 0; k < kJT; ++k) accumulate(ST + k * kRT + rbase, Xs[k * P + pcol]);
        __syncthreads();
    }

    // Off-diagonal blocks: e^{cum_i} C_i^T h_{c-1}, with the decay folded into C (transposed)
    for (int e = tid; e < N * kRT; e += kThreads) {
        const int n = e / kRT, r = e % kRT;
        const int i = i0 + r;
        CT[n * kRT + r] = (i < L) ? Cs[r * NS + n] * dexp<IO>(As[n] * lcum[i]) : 0.f;
    }
    const float *hprev = w.states + (((int64_t)bi * p.H + h) * p.nc + c) * N * P;
    for (int nb0 = 0; nb0 < N; nb0 += kJT) {
        __syncthreads();
        load_tile(Hs, P, hprev, (int64_t)nb0 * P, (int64_t)P, kJT, N - nb0, P);
        __syncthreads();
        const int kmax = min(kJT, N - nb0);
        if (active)
            for (int k = 0; k < kmax; ++k) accumulate(CT + (nb0 + k) * kRT + rbase, Hs[k * P + pcol]);
    }

    IO *Y = static_cast<IO *>(p.y);
    const float Dh = p.D ? p.D[h] : 0.f;
    if (active) {
#pragma unroll
        for (int a = 0; a < kMaxOut; ++a) {
            const int i = i0 + rbase + a;
            if (a < nout && i < L) {
                const int64_t off = (((int64_t)bi * p.T + t0 + i) * p.H + h) * P + pcol;
                float v = acc[a];
                if (p.D) v = fmaf(Dh, ld_io(X, off), v);
                st_io(Y, off, v);
            }
        }
    }
}

size_t state_smem(const Problem &p) { return sizeof(float) * (((p.Q + 3) & ~3) + kTT * ((p.N + 3) & ~3) + kTT * p.P); }
size_t output_smem(const Problem &p) {
    const size_t NS = p.N + 1;
    return sizeof(float) * (p.Q + p.N + kRT * NS + kJT * NS + kJT * p.P + 3 + kJT * kRT + p.N * kRT);
}

template <typename IO, int ACC>
cudaError_t launch_state(const Problem &p, const GenericWorkspace &w, cudaStream_t s) {
    const size_t sm1 = state_smem(p);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gen_chunk_state<IO, ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm1)) != cudaSuccess)
        return e;
    dim3 g1((unsigned)p.nc, (unsigned)p.H, (unsigned)p.b);
    gen_chunk_state<IO, ACC><<<g1, kThreads, sm1, s>>>(p, w);
    return cudaGetLastError();
}

// The first two kernels: chunk states, then the states entering every chunk (in place).
template <typename IO>
cudaError_t launch_states(const Problem &p, const GenericWorkspace &w, cudaStream_t s) {
    cudaError_t e;
    // accumulators per thread of the chunk-state kernel: N / (threads / P), rounded up
    const int64_t nacc = (p.N + (kThreads / p.P) - 1) / (kThreads / p.P);
    if (nacc <= 4) e = launch_state<IO, 4>(p, w, s);
    else if (nacc <= 8) e = launch_state<IO, 8>(p, w, s);
    else if (nacc <= 16) e = launch_state<IO, 16>(p, w, s);
    else if (nacc <= 32) e = launch_state<IO, 32>(p, w, s);
    else e = launch_state<IO, kMaxAcc>(p, w, s);
    if (e != cudaSuccess) return e;
    dim3 g2((unsigned)((p.N * p.P + kThreads - 1) / kThreads), (unsigned)p.H, (unsigned)p.b);
    gen_state_passing<<<g2, kThreads, 0, s>>>(p, w);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_typed(const Problem &p, const GenericWorkspace &w, cudaStream_t s) {
    const size_t sm3 = output_smem(p);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gen_chunk_output<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sm3)) != cudaSuccess)
        return e;
    if ((e = launch_states<IO>(p, w, s)) != cudaSuccess) return e;
    const int64_t nrt = (p.Q + kRT - 1) / kRT;
    dim3 g3((unsigned)(p.nc * nrt), (unsigned)p.H, (unsigned)p.b);
    record_dominant_start(s);
    gen_chunk_output<IO><<<g3, kThreads, sm3, s>>>(p, w);
    record_dominant_stop(s);
    note_launches(3);
    return cudaGetLastError();
}

}  // namespace

bool generic_supports(const Problem &p) {
    if (p.P < 1 || p.P > 256 || (p.P & (p.P - 1))) return false;
    // launch limits of the three grids: (chunks [x 32-row tiles], H, b)
    if (p.H > 65535 || p.b > 65535) return false;
    if (p.nc * ((p.Q + kRT - 1) / kRT) > (int64_t)INT32_MAX) return false;
    if (p.N < 1 || p.N > 256 || p.N * p.P > (int64_t)kMaxAcc * kThreads) return false;
    if (p.Q > kThreads) return false;
    if (kRT * p.P > (int64_t)kMaxOut * kThreads) return false;
    return output_smem(p) <= 227 * 1024;
}

size_t generic_workspace_bytes(const Problem &p) {
    size_t off = kStatusBytes;
    off += align_up(sizeof(float) * (size_t)(p.b * p.H * p.nc), 256);
    off += sizeof(float) * (size_t)(p.b * p.H * p.nc * p.N * p.P);
    return off;
}

GenericWorkspace generic_carve(const Problem &p, void *ws) {
    char *base = static_cast<char *>(ws);
    GenericWorkspace w;
    w.status = reinterpret_cast<int *>(base);
    w.chunk_sum = reinterpret_cast<float *>(base + kStatusBytes);
    w.states = reinterpret_cast<float *>(base + kStatusBytes +
                                         align_up(sizeof(float) * (size_t)(p.b * p.H * p.nc), 256));
    return w;
}

cudaError_t generic_launch(const Problem &p, const GenericWorkspace &w, cudaStream_t s) {
    if (p.io_dtype == SSD_DTYPE_BF16) return launch_typed<__nv_bfloat16>(p, w, s);
    return launch_typed<float>(p, w, s);
}

cudaError_t generic_passing_launch(const Problem &p, const GenericWorkspace &w, cudaStream_t s) {
    dim3 g2((unsigned)((p.N * p.P + kThreads - 1) / kThreads), (unsigned)p.H, (unsigned)p.b);
    gen_state_passing<<<g2, kThreads, 0, s>>>(p, w);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssd
