// ssd_scan.cu -- the linear form of the selective recurrence on CUDA cores.
//
// The same map as ssd_fwd, evaluated token by token instead of by the chunked
// algorithm: for each (batch row, head),
//
//   h_t = a_t (.) h_{t-1} + B_t x_t^T        (N x P state, fp32)
//   y_t = C_t^T h_t + D x_t
//
// (Structured State Space Duality, "The recurrence as one matrix": the linear
// O(T) form.  Its intro describes the earlier selective-scan kernels that ran
// this recurrence elementwise on the general-purpose units; the chunked form
// moves most of the work onto tensor cores instead.)  This kernel is that
// elementwise form: the decode step of a served model (one token, state in
// place) and the comparison the pages draw between the two forms.
//
// One CTA per (batch row, head); the state lives in registers for the whole
// sequence.  Thread t owns state column p = t mod P and the NS consecutive
// state rows of slice s = t / P (S = 256 / P slices; NS a multiple of 4, the
// rows past N padded with zeros).  Tokens are staged 32 at a time in shared
// memory (x, B and C rows padded to S NS entries, and the decay); every thread
// updates its state entries, reading B and C four rows at a time (a broadcast
// within the warp), accumulates its slice's partial C_t^T h_t in four
// independent sums, and the slices' partials are summed once per chunk.
#include <cuda_bf16.h>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kScanThreads = 256;
constexpr int kTC = 32;            // tokens per staged chunk

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
// e^x of a decay: fp32 io keeps expf (its tolerance is 1e-5); bf16 io (tolerance 2e-3) the
// hardware base-2 exponential (relative error ~2^-22).
template <typename IO> __device__ __forceinline__ float dexp(float x);
template <> __device__ __forceinline__ float dexp<float>(float x) { return expf(x); }
template <> __device__ __forceinline__ float dexp<__nv_bfloat16>(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

// State rows per thread: the smallest instantiated width (4, 8, 16, 32 or 64) that covers
// ceil(N / S); 0 when none does.
int64_t scan_rows(const Problem &p) {
    const int64_t S = kScanThreads / p.P;
    const int64_t need = (p.N + S - 1) / S;
    for (int64_t k = 4; k <= 64; k *= 2)
        if (need <= k) return k;
    return 0;
}

size_t scan_smem(const Problem &p) {
    const int64_t S = kScanThreads / p.P;
    const int64_t NP = S * scan_rows(p);
    // x [kTC][P], B and C [kTC][NP], decay [kTC] (scalar A) or dt [kTC] (diagonal A), partials [kTC][S][P]
    return sizeof(float) * (size_t)(kTC * (p.P + 2 * NP + 4) + kTC * S * p.P);
}

template <typename IO, bool kDiag, int NS>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(Problem p) {
    extern __shared__ float sm[];
    const int P = (int)p.P, N = (int)p.N, H = (int)p.H;
    const int S = kScanThreads / P;
    const int NP = S * NS;                 // padded row length of the staged B and C
    const int tid = threadIdx.x;
    const int pp = tid % P, sl = tid / P;
    const int bi = blockIdx.x / H, h = blockIdx.x % H;
    const int g = h / (H / (int)p.G);
    const int64_t T = p.T;
    float *xs = sm;                       // [kTC][P]
    float *Bs = xs + kTC * P;             // [kTC][NP]
    float *Cs = Bs + kTC * NP;            // [kTC][NP]
    float *ds = Cs + kTC * NP;            // [kTC] (+3 for alignment)
    float *part = ds + kTC + 4;           // [kTC][S][P]
    const IO *X = static_cast<const IO *>(p.x);
    const IO *Bm = static_cast<const IO *>(p.B);
    const IO *Cm = static_cast<const IO *>(p.C);
    IO *Y = static_cast<IO *>(p.y);
    const int64_t sidx = (int64_t)bi * H + h;

    float hs[NS];
    float An[kDiag ? NS : 1];
#pragma unroll
    for (int e = 0; e < NS; ++e) {
        const int n = sl * NS + e;
        hs[e] = (p.init && n < N) ? p.init[(sidx * N + n) * P + pp] : 0.f;
        if constexpr (kDiag) An[e] = (n < N) ? p.A[(int64_t)h * N + n] : 0.f;
    }
    const float Ah = kDiag ? 0.f : p.A[h];
    const float Dh = p.D ? p.D[h] : 0.f;

    for (int64_t t0 = 0; t0 < T; t0 += kTC) {
        const int L = (int)min((int64_t)kTC, T - t0);
        __syncthreads();                  // the previous chunk's partials have been summed
        for (int i = tid; i < L * P; i += kScanThreads) {
            const int tt = i / P, c = i % P;
            xs[i] = ld_io(X, ((int64_t)bi * T + t0 + tt) * H * P + (int64_t)h * P + c);
        }
        for (int i = tid; i < L * NP; i += kScanThreads) {
            const int tt = i / NP, c = i % NP;
            const int64_t off = ((int64_t)bi * T + t0 + tt) * p.G * N + (int64_t)g * N + c;
            Bs[i] = c < N ? ld_io(Bm, off) : 0.f;
            Cs[i] = c < N ? ld_io(Cm, off) : 0.f;
        }
        for (int i = tid; i < L; i += kScanThreads) {
            const float d = p.dt[((int64_t)bi * T + t0 + i) * H + h];
            ds[i] = kDiag ? d : dexp<IO>(d * Ah);   // scalar A: the token's decay a_t itself
        }
        __syncthreads();
        for (int tt = 0; tt < L; ++tt) {
            const float xv = xs[tt * P + pp];
            const float dv = ds[tt];
            const float4 *b4 = reinterpret_cast<const float4 *>(Bs + tt * NP + sl * NS);
            const float4 *c4 = reinterpret_cast<const float4 *>(Cs + tt * NP + sl * NS);
            float yq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e4 = 0; e4 < NS / 4; ++e4) {
                const float4 bv = b4[e4], cv = c4[e4];
                const float bb[4] = {bv.x, bv.y, bv.z, bv.w}, cc[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = 4 * e4 + u;
                    const float a = kDiag ? dexp<IO>(dv * An[e]) : dv;
                    hs[e] = fmaf(a, hs[e], bb[u] * xv);
                    yq[u] = fmaf(cc[u], hs[e], yq[u]);
                }
            }
            part[(tt * S + sl) * P + pp] = (yq[0] + yq[1]) + (yq[2] + yq[3]);
        }
        __syncthreads();
        for (int i = tid; i < L * P; i += kScanThreads) {
            const int tt = i / P, c = i % P;
            float yv = Dh * xs[i];
            for (int s2 = 0; s2 < S; ++s2) yv += part[(tt * S + s2) * P + c];
            st_io(Y, ((int64_t)bi * T + t0 + tt) * H * P + (int64_t)h * P + c, yv);
        }
    }
    if (p.final_state) {
#pragma unroll
        for (int e = 0; e < NS; ++e) {
            const int n = sl * NS + e;
            if (n < N) p.final_state[(sidx * N + n) * P + pp] = hs[e];
        }
    }
}

// One token (T = 1: the decode step, and ssd_scan at T = 1): the state read and written in
// 16-byte pieces.  One CTA per (batch row, head), 256 threads; thread t updates the float4s
// e = t + 256 k of the N x P/4 state (row e / (P/4), columns 4 (e mod P/4) ..), all in the same
// columns, so its part of C^T h is four sums; the parts are summed over a warp's rows by
// shuffles and over the warps through shared memory.
constexpr int kDecThreads = 256;

template <typename IO, bool kDiag>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(Problem p) {
    __shared__ float sB[256], sC[256], sa[256];
    __shared__ float sx[256], part[kDecThreads / 32][256];
    const int P = (int)p.P, N = (int)p.N, H = (int)p.H;
    const int P4 = P / 4;
    const int bi = blockIdx.x / H, h = blockIdx.x % H;
    const int g = h / (H / (int)p.G);
    const int64_t sidx = (int64_t)bi * H + h;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float dtv = p.dt[(int64_t)bi * H + h];
    for (int i = tid; i < N; i += kDecThreads) {
        const int64_t off = ((int64_t)bi * p.G + g) * N + i;
        sB[i] = ld_io(static_cast<const IO *>(p.B), off);
        sC[i] = ld_io(static_cast<const IO *>(p.C), off);
        sa[i] = kDiag ? expf(dtv * p.A[(int64_t)h * N + i]) : 0.f;
    }
    for (int i = tid; i < P; i += kDecThreads) sx[i] = ld_io(static_cast<const IO *>(p.x), sidx * P + i);
    const float a_s = kDiag ? 0.f : expf(dtv * p.A[h]);
    __syncthreads();
    const int p4 = tid % P4;
    float x4[4], y4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) x4[j] = sx[4 * p4 + j];
    const float4 *src = p.init ? reinterpret_cast<const float4 *>(p.init + sidx * N * P) : nullptr;
    float4 *dst = reinterpret_cast<float4 *>(p.final_state + sidx * N * P);
    for (int e = tid; e < N * P4; e += kDecThreads) {
        const int n = e / P4;
        const float a = kDiag ? sa[n] : a_s, bn = sB[n], cn = sC[n];
        const float4 hv = src ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 nv = make_float4(fmaf(a, hv.x, bn * x4[0]), fmaf(a, hv.y, bn * x4[1]),
                                      fmaf(a, hv.z, bn * x4[2]), fmaf(a, hv.w, bn * x4[3]));
        dst[e] = nv;
        y4[0] = fmaf(cn, nv.x, y4[0]);
        y4[1] = fmaf(cn, nv.y, y4[1]);
        y4[2] = fmaf(cn, nv.z, y4[2]);
        y4[3] = fmaf(cn, nv.w, y4[3]);
    }
    // lanes P4 apart hold the same columns
    for (int o = P4; o < 32; o <<= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) y4[j] += __shfl_xor_sync(0xffffffffu, y4[j], o);
    }
    if (lane < P4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) part[warp][4 * lane + j] = y4[j];
    }
    __syncthreads();
    const float Dh = p.D ? p.D[h] : 0.f;
    for (int c = tid; c < P; c += kDecThreads) {
        float acc = Dh * sx[c];
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) acc += part[w][c];
        st_io(static_cast<IO *>(p.y), sidx * P + c, acc);
    }
}

// The one-token kernel applies: 4 <= P <= 128 (a row's columns within one warp), N <= 256, and
// 16-byte aligned states.
bool decode_applies(const Problem &p) {
    if (p.T != 1 || !p.final_state || p.P < 4 || p.P > 128 || p.N > 256) return false;
    if ((reinterpret_cast<uintptr_t>(p.final_state) & 15u) != 0) return false;
    if (p.init && (reinterpret_cast<uintptr_t>(p.init) & 15u) != 0) return false;
    return true;
}

template <typename IO, bool kDiag>
cudaError_t launch_ns(const Problem &p, cudaStream_t s) {
    const int64_t ns = scan_rows(p);
    const size_t smem = scan_smem(p);
    const unsigned grid = (unsigned)(p.b * p.H);
#define SSD_SCAN_CASE(K)                                                                                  \
    if (ns == K) {                                                                                        \
        cudaError_t e = cudaFuncSetAttribute(scan_kernel<IO, kDiag, K>,                                   \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
        if (e != cudaSuccess) return e;                                                                   \
        record_dominant_start(s);                                                                         \
        scan_kernel<IO, kDiag, K><<<grid, kScanThreads, smem, s>>>(p);                                    \
        record_dominant_stop(s);                                                                          \
        note_launches(1);                                                                                 \
        return cudaGetLastError();                                                                        \
    }
    SSD_SCAN_CASE(4)
    SSD_SCAN_CASE(8)
    SSD_SCAN_CASE(16)
    SSD_SCAN_CASE(32)
    SSD_SCAN_CASE(64)
#undef SSD_SCAN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool scan_supports(const Problem &p) {
    if (p.P < 1 || p.P > kScanThreads || (p.P & (p.P - 1))) return false;
    if (scan_rows(p) == 0) return false;                  // state entries per thread
    if (p.b * p.H > (int64_t)INT32_MAX) return false;     // one CTA per (batch row, head)
    return scan_smem(p) <= 227 * 1024;
}

cudaError_t scan_launch(const Problem &p, cudaStream_t s) {
    const bool diag = p.a_mode == SSD_A_DIAGONAL;
    if (decode_applies(p)) {
        const unsigned grid = (unsigned)(p.b * p.H);
        record_dominant_start(s);
        if (p.io_dtype == SSD_DTYPE_BF16) {
            if (diag) decode_kernel<__nv_bfloat16, true><<<grid, kDecThreads, 0, s>>>(p);
            else decode_kernel<__nv_bfloat16, false><<<grid, kDecThreads, 0, s>>>(p);
        } else {
            if (diag) decode_kernel<float, true><<<grid, kDecThreads, 0, s>>>(p);
            else decode_kernel<float, false><<<grid, kDecThreads, 0, s>>>(p);
        }
        record_dominant_stop(s);
        note_launches(1);
        return cudaGetLastError();
    }
    if (p.io_dtype == SSD_DTYPE_BF16)
        return diag ? launch_ns<__nv_bfloat16, true>(p, s) : launch_ns<__nv_bfloat16, false>(p, s);
    return diag ? launch_ns<float, true>(p, s) : launch_ns<float, false>(p, s);
}

}  // namespace ssd
