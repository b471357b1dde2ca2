// ssd_diag_tc.cu -- the SSD forward pass with a diagonal A on tcgen05 tensor
// cores (sm_103a): TMA tile loads, tcgen05.mma with TMEM accumulators, the
// state kept in TMEM for the whole sequence.
//
// With a diagonal A every state dimension n decays at its own rate
// (Structured State Space Duality, "What the duality gives up"; On Structured
// State-Space Duality, abstract, point (i)), so the masked matrix of a chunk no
// longer factors as (C B^T) o L.  Over a block of 128 tokens, with Dt_t the
// inclusive prefix sum of dt inside the block and the decay of dimension n
// between tokens j <= i equal to exp(A_n (Dt_i - Dt_j)):
//
//   y_i = sum_{j <= i} S_ij x_j + sum_n C_in exp(A_n Dt_i) h_prev[n, :]  (+ D x_i)
//   S_ij = sum_n C_in B_jn exp(A_n (Dt_i - Dt_j))
//   h = exp(A Dt_end) o h_prev + sum_j (B_j o exp(A (Dt_end - Dt_j))) x_j^T
//
// The block's rows fall into eight 16-token groups; R_J is Dt at the last token
// of group J (R_{-1} = 0) and M_J at its eighth token.  Every product is split
// at a reference point between its two tokens, so that each factor carried by a
// tensor-core operand is <= 1 (fp16 operands, fp32 accumulation):
//
//  * S_ij, j in group J < group I of i: exp(A (Dt_i - R_J)) on the C side and
//    exp(A (R_J - Dt_j)) on the B side.  The C side depends on J, so every row
//    keeps one copy of its decayed C per earlier group -- written to TMEM, where
//    the MMA takes it as its A operand -- and the seven products
//    copy_J (128 x 64) x B~_J^T (64 x 16) fill S's columns group by group.
//  * S_ij, j and i in the same group: on the CUDA cores in fp32, split at M_I
//    (factors up to exp(|A| x half the group's Dt range); a group whose factors
//    could leave fp32 takes one exponential per (i, j, n) instead).
//  * h_prev enters through C o exp(A Dt_i) (in TMEM) x h_prev (fp16, shared memory);
//    the state's own product B o w (w <= 1) accumulates onto exp(A Dt_end) o h_prev,
//    which the rows of the state rescale in place in TMEM.
//
// The same map as the chunked algorithm of the other paths (equal up to
// rounding); the block of 128 tokens plays the chunk's part whatever Q is.
//
// One CTA per (batch row, head) at a time (persistent over sequences), 6 warps:
//   warp 0      TMA producer: X, B, C tiles of a block (two stages)
//   warp 1      TMEM owner; lane 0 issues every MMA
//   warps 2-5   math: thread = TMEM lane = row i of the block (warp w owns lanes
//               32 (w mod 4) ...); rows 0-63 also own the state rows n = i.
// TMEM (512 columns): S 0-127 (fp32; its fp16 form overwrites columns 0-63 as it
// is read), C copies 128-351 (7 x 32, fp16 pairs), C o exp(A Dt) 352-383, Y
// 384-447, h 448-511 (lanes 0-63).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "ssd_internal.cuh"
#include "ssd_ptx.cuh"

namespace ssd {
namespace {

using namespace ptx;

constexpr int kBlk = 128;          // tokens per block
constexpr int kP = 64;             // head dim of this path
constexpr int kN = 64;             // state dim of this path
constexpr int kThreads = 192;      // 6 warps
constexpr int kTile = 128 * 128;   // 128 rows x 64 16-bit values

// shared memory (byte offsets from a 1024-aligned base)
constexpr int kStageBytes = 3 * kTile;                 // X, B, C (bf16 as loaded; X then fp16)
constexpr int kOffStage = 0;                           // [2 stages]
constexpr int kOffBt = 2 * kStageBytes;                // B~ (fp16, [j][n], 128B swizzle)
constexpr int kOffBw = kOffBt + kTile;                 // B o w (fp16, [j][n])
constexpr int kOffBp = kOffBw + kTile;                 // B' (fp32, [j][64]) for the diagonal groups
constexpr int kOffHp = kOffBp + 2 * kTile;             // h_prev (fp16, [n][p])
constexpr int kOffY = kOffHp + 64 * 128;               // y: [4 warps][32 rows][128 B]
constexpr int kTabRow = 68;                            // floats per table row (64 + bank padding)
constexpr int kTabRows = 22;                           // per warp: T1 T2 T3 T5 x 2 groups, G x 2 groups x 7
constexpr int kTabWarpBytes = kTabRows * kTabRow * 4;
constexpr int kOffTab = kOffY + kTile;                 // per-warp tables
constexpr int kOffDtW = kOffTab + 4 * kTabWarpBytes;   // per-warp Dt of all 128 rows
constexpr int kOffA2 = kOffDtW + 4 * 512;              // per-warp A (log2 units), 64 floats
constexpr int kOffMisc = kOffA2 + 4 * 256;             // TMEM base, abort flag
constexpr int kOffBar = kOffMisc + 16;
constexpr int kNumBars = 8;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;   // + alignment slack

constexpr int B_FULL = 0;     // [2] TMA landed a stage
constexpr int B_EMPTY = 2;    // [2] the math warps are done with a stage (4 warps)
constexpr int B_OPS = 4;      // operands of a block written (4 warps)
constexpr int B_SFULL = 5;    // S, Y_off and the state product are done
constexpr int B_S16 = 6;      // S (fp16) written (4 warps)
constexpr int B_YFULL = 7;    // S X is done

constexpr uint32_t kTmS = 0;
constexpr uint32_t kTmS16 = 0;
constexpr uint32_t kTmCp = 128;
constexpr uint32_t kTmCh = 352;
constexpr uint32_t kTmY = 384;
constexpr uint32_t kTmH = 448;

// Factors exp2(a) with |a| up to this stay inside fp32 (normal) range.
constexpr float kSafeLog2 = 110.f;

struct DiagParams {
    const float *dt, *A, *D, *init;
    float *final_state;
    int *status;
    int b, T, H, G, nblk, nseq;
};

// The diagonal group of a row whose split factors could leave fp32: S_ij =
// sum_n C_in B_jn exp(A_n (Dt_i - Dt_j)) with one exponential per term (C from the
// row's tile, B from the B' table, which holds B itself for such a group).
static __device__ __noinline__ void diag_group_direct(const unsigned char *crow, uint32_t rx, const float *Bp,
                                                      const float *A2s, const float *DtW, int i, float *d) {
    const int I = i >> 4, sw = I & 1;
    const float Dti = DtW[i];
    float c[64];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        const uint4 w = *reinterpret_cast<const uint4 *>(crow + ((16u * cc) ^ rx));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = bf2_to_f2(ws[e]);
            c[8 * cc + 2 * e] = f.x;
            c[8 * cc + 2 * e + 1] = f.y;
        }
    }
    for (int jj = 0; jj < 16; ++jj) {
        const int j = 16 * I + jj;
        const float4 *brow = reinterpret_cast<const float4 *>(Bp + j * 64);
        const float dd = Dti - DtW[j];
        float s0 = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
            const float4 bv = brow[c4 ^ sw];
            const int n = 4 * c4;
            s0 = fmaf(c[n] * bv.x, ex2(A2s[n] * dd), s0);
            s0 = fmaf(c[n + 1] * bv.y, ex2(A2s[n + 1] * dd), s0);
            s0 = fmaf(c[n + 2] * bv.z, ex2(A2s[n + 2] * dd), s0);
            s0 = fmaf(c[n + 3] * bv.w, ex2(A2s[n + 3] * dd), s0);
        }
        d[jj] = jj <= (i & 15) ? s0 : 0.f;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    ssd_diag_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                    const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y,
                    const DiagParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
    const Ctl ctl{p.status, abort_flag};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 4);
        }
        mbar_init(bar(B_OPS), 4);
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_S16), 4);
        mbar_init(bar(B_YFULL), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int hpg = p.H / p.G;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int kb = 0;
            bool ok = true;
            for (int sq = blockIdx.x; sq < p.nseq && ok; sq += gridDim.x) {
                const int bi = sq / p.H, h = sq - bi * p.H, g = h / hpg;
                for (int c = 0; c < p.nblk; ++c, ++kb) {
                    const int st = kb & 1;
                    if (kb >= 2 && !(ok = wait_bar(ctl, bar(B_EMPTY + st), ((kb >> 1) - 1) & 1))) break;
                    const uint32_t dst = sbase + kOffStage + st * kStageBytes;
                    mbar_expect_tx(bar(B_FULL + st), 3 * kTile);
                    tma_load_3d(dst, &tm_x, bar(B_FULL + st), h * kP, c * kBlk, bi);
                    tma_load_3d(dst + kTile, &tm_B, bar(B_FULL + st), g * kN, c * kBlk, bi);
                    tma_load_3d(dst + 2 * kTile, &tm_C, bar(B_FULL + st), g * kN, c * kBlk, bi);
                }
            }
            // after an abort: wait (bounded) for the loads still in flight
            if (!ok)
                for (int k2 = kb - 2; k2 < kb; ++k2)
                    if (k2 >= 0) drain_bar(bar(B_FULL + (k2 & 1)), (k2 >> 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_f16(128, 16, 0, 0);    // copy_J x B~_J^T
            const uint32_t id_y = idesc_f16(128, kP, 0, 1);    // (C o e) h_prev, S X
            const uint32_t id_st = idesc_f16(128, kP, 1, 1);   // (B o w)^T X
            const bool has_d = p.D != nullptr;
            // B~: K-major, rows of group J at +2048 J bytes; K steps of 16: +32 bytes
            const uint64_t dbt = sdesc(sbase + kOffBt, 16, 1024);
            // B o w as the MN-major A of the state product: M = 128 in two 64-wide atoms; the
            // second (rows 64-127 of the product, never read) points at the B' table
            const uint64_t dbw = sdesc(sbase + kOffBw, kTile, 1024);
            const uint64_t dhp = sdesc(sbase + kOffHp, kTile, 1024);
            int kb = 0;
            uint32_t last_bar = 0, last_par = 0;   // the last commit issued (0: none)
            bool ok = true;
            for (int sq = blockIdx.x; sq < p.nseq && ok; sq += gridDim.x) {
                for (int c = 0; c < p.nblk; ++c, ++kb) {
                    const int st = kb & 1;
                    const uint64_t dx = sdesc(sbase + kOffStage + st * kStageBytes, kTile, 1024);
                    if (!(ok = wait_bar(ctl, bar(B_OPS), kb & 1))) break;
                    tc_fence_after();
                    for (int J = 0; J < 7; ++J)
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(tmem + kTmS + 16 * J, tmem + kTmCp + 32 * J + 8 * kk,
                                   dbt + (uint64_t)(128 * J + 2 * kk), id_s, kk > 0);
                    for (int kk = 0; kk < 4; ++kk)   // K = n: steps of 16 rows of h_prev (+2048 bytes)
                        mma_ts(tmem + kTmY, tmem + kTmCh + 8 * kk, dhp + (uint64_t)(128 * kk), id_y,
                               (kk > 0) || has_d);
                    for (int kk = 0; kk < 8; ++kk)   // K = tokens: steps of 16 rows (+2048 bytes)
                        mma_ss(tmem + kTmH, dbw + (uint64_t)(128 * kk), dx + (uint64_t)(128 * kk), id_st, 1);
                    mma_commit(bar(B_SFULL));
                    last_bar = bar(B_SFULL);
                    last_par = kb & 1;
                    if (!(ok = wait_bar(ctl, bar(B_S16), kb & 1))) break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tmem + kTmY, tmem + kTmS16 + 8 * kk, dx + (uint64_t)(128 * kk), id_y, 1);
                    mma_commit(bar(B_YFULL));
                    last_bar = bar(B_YFULL);
                    last_par = kb & 1;
                }
            }
            // after an abort: let the products in flight finish before TMEM is freed
            if (!ok && last_bar) drain_bar(last_bar, last_par);
        }
    } else {
        // ------------------------------------------------------------ math warps
        const int q = warp & 3;                     // TMEM lane quarter
        const int i = 32 * q + lane;                // row of the block (token / state row)
        const int I = i >> 4;                       // 16-row group
        const int lg = (lane >> 4) & 1;             // the group's index within this warp
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        float *tab = reinterpret_cast<float *>(smem + kOffTab + q * kTabWarpBytes);
        float *DtW = reinterpret_cast<float *>(smem + kOffDtW + q * 512);
        float *A2s = reinterpret_cast<float *>(smem + kOffA2 + q * 256);
        float *Bp = reinterpret_cast<float *>(smem + kOffBp);
        unsigned char *ybuf = smem + kOffY + q * 4096;
        const uint32_t ybuf_a = sbase + kOffY + q * 4096;
        // Every table factor lies in (0, 1]; those that multiply a factor above 1 (T1, T5) are
        // at least 2^-110 in a group within the split's range, so no product underflows
        // unless its exact value is below fp32's normal range.
        auto T1 = [&](int n) -> float & { return tab[(0 + lg) * kTabRow + n]; };   // exp(A (M_I - R_{I-1}))
        auto T2 = [&](int n) -> float & { return tab[(2 + lg) * kTabRow + n]; };   // exp(A R_{I-1})
        auto T3 = [&](int n) -> float & { return tab[(4 + lg) * kTabRow + n]; };   // exp(A (Dt_end - R_I))
        auto T5 = [&](int n) -> float & { return tab[(6 + lg) * kTabRow + n]; };   // exp(A (R_I - M_I))
        auto Gt = [&](int J, int n) -> float & { return tab[(8 + 7 * lg + J) * kTabRow + n]; };  // exp(A (R_{I-1} - R_J))
        uint32_t bad = 0;
        int kb = 0;
        for (int sq = blockIdx.x; sq < p.nseq; sq += gridDim.x) {
            const int bi = sq / p.H, h = sq - bi * p.H;
            __syncwarp();
            const float a0 = p.A[(int64_t)h * kN + lane] * kLog2e, a1 = p.A[(int64_t)h * kN + 32 + lane] * kLog2e;
            A2s[lane] = a0;
            A2s[32 + lane] = a1;
            float amax = fmaxf(fabsf(a0), fabsf(a1));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float Dh = p.D ? p.D[h] : 0.f;
            __syncwarp();
            // the initial state into TMEM (state rows 0-63: quarters 0 and 1)
            if (q < 2) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float v[32];
                    const float *src = p.init ? p.init + ((int64_t)sq * kN + i) * kP + 32 * half : nullptr;
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 f = src ? __ldg(reinterpret_cast<const float4 *>(src + e))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[e] = f.x;
                        v[e + 1] = f.y;
                        v[e + 2] = f.z;
                        v[e + 3] = f.w;
                    }
                    tmem_st32(tmem + lane_off + kTmH + 32 * half, v);
                }
                tmem_st_wait();
            }
            auto load_dt = [&](int c, float (&v)[4]) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = c * kBlk + 32 * m + lane;
                    v[m] = t < p.T ? __ldg(p.dt + ((int64_t)bi * p.T + t) * p.H + h) : 0.f;
                }
            };
            float dtn[4];
            load_dt(0, dtn);
            for (int c = 0; c < p.nblk; ++c, ++kb) {
                const int st = kb & 1;
                // (1) Dt: inclusive prefix sums of dt over the block (four interleaved 32-row
                // scans; every warp computes all 128 rows), the warp's tables
                float Dv[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) Dv[m] = dtn[m];
                if (c + 1 < p.nblk) load_dt(c + 1, dtn);
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float u = __shfl_up_sync(0xffffffffu, Dv[m], o);
                        if (lane >= o) Dv[m] += u;
                    }
                }
                {
                    float run = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float tot = __shfl_sync(0xffffffffu, Dv[m], 31);
                        Dv[m] += run;
                        run += tot;
                    }
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) DtW[32 * m + lane] = Dv[m];
                __syncwarp();
                const float Dti = DtW[i];
                const float Dend = DtW[127];
                const float RI = DtW[16 * I + 15], MI = DtW[16 * I + 7];
                const float Rm1 = I > 0 ? DtW[16 * I - 1] : 0.f;
                const bool safe = amax * fmaxf(MI - Rm1, RI - MI) <= kSafeLog2;
                // tables of this warp's two groups: T1, T2, T3, T5 and G (per earlier group J)
#pragma unroll
                for (int hn = 0; hn < 2; ++hn) {
                    const int n = lane + 32 * hn;
                    const float an = hn ? a1 : a0;
#pragma unroll
                    for (int l2 = 0; l2 < 2; ++l2) {
                        const int I2 = 2 * q + l2;
                        const float r1 = I2 > 0 ? DtW[16 * I2 - 1] : 0.f;
                        const float m2 = DtW[16 * I2 + 7], r2 = DtW[16 * I2 + 15];
                        tab[(0 + l2) * kTabRow + n] = ex2(an * (m2 - r1));
                        tab[(2 + l2) * kTabRow + n] = ex2(an * r1);
                        tab[(4 + l2) * kTabRow + n] = ex2(an * (Dend - r2));
                        tab[(6 + l2) * kTabRow + n] = ex2(an * (r2 - m2));
                    }
#pragma unroll
                    for (int l2 = 0; l2 < 2; ++l2) {
                        const int I2 = 2 * q + l2;
                        const float r1 = I2 > 0 ? DtW[16 * I2 - 1] : 0.f;
                        for (int J = 0; J < I2; ++J) tab[(8 + 7 * l2 + J) * kTabRow + n] = ex2(an * (r1 - DtW[16 * J + 15]));
                    }
                }
                __syncwarp();

                // (2) state rows: h_prev (fp16) for (C o e) h_prev; h <- exp(A Dt_end) o h in place
                if (q < 2) {
                    const float an = ex2(A2s[i] * Dend);
                    unsigned char *hrow = smem + kOffHp + i * 128;
                    const uint32_t rx = (uint32_t)(i & 7) * 16u;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float hv[32];
                        tmem_ld32(tmem + lane_off + kTmH + 32 * half, hv);
                        tmem_ld_wait();
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int e = 8 * cc;
                            *reinterpret_cast<uint4 *>(hrow + ((16u * (4 * half + cc)) ^ rx)) =
                                make_uint4(pack_h2(hv[e], hv[e + 1]), pack_h2(hv[e + 2], hv[e + 3]),
                                           pack_h2(hv[e + 4], hv[e + 5]), pack_h2(hv[e + 6], hv[e + 7]));
                        }
#pragma unroll
                        for (int e = 0; e < 32; ++e) hv[e] *= an;
                        tmem_st32(tmem + lane_off + kTmH + 32 * half, hv);
                    }
                }

                // (3) operands of row i
                wait_bar(ctl, bar(B_FULL + st), (kb >> 1) & 1);
                unsigned char *xt = smem + kOffStage + st * kStageBytes;
                const uint32_t rx = (uint32_t)(i & 7) * 16u;
                {
                    // X: bf16 -> fp16 in place; D x into Y's columns (Y_off accumulates onto it)
                    unsigned char *row = xt + i * 128;
                    uint4 u[8];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) u[cc] = *reinterpret_cast<const uint4 *>(row + ((16u * cc) ^ rx));
                    if (p.D) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            float dx[32];
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc) {
                                const uint4 w = u[4 * half + cc];
                                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = bf2_to_f2(ws[e]);
                                    dx[8 * cc + 2 * e] = Dh * f.x;
                                    dx[8 * cc + 2 * e + 1] = Dh * f.y;
                                }
                            }
                            tmem_st32(tmem + lane_off + kTmY + 32 * half, dx);
                        }
                    }
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        u[cc].x = bf2_to_h2(u[cc].x);
                        u[cc].y = bf2_to_h2(u[cc].y);
                        u[cc].z = bf2_to_h2(u[cc].z);
                        u[cc].w = bf2_to_h2(u[cc].w);
                        *reinterpret_cast<uint4 *>(row + ((16u * cc) ^ rx)) = u[cc];
                    }
                }
                {
                    // B: B' = B exp(A (M_I - Dt_i)) (fp32, for the diagonal group), B~ = B' T5 =
                    // B exp(A (R_I - Dt_i)), B o w = B~ T3 = B exp(A (Dt_end - Dt_i)) (fp16); a group
                    // outside the split's range keeps B itself in B' and forms B~ directly
                    const unsigned char *row = xt + kTile + i * 128;
                    float *bprow = Bp + i * 64;
                    const int sw = I & 1;
#pragma unroll 2
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + ((16u * cc) ^ rx));
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                        float bv[8], bt[8], bw[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = bf2_to_f2(ws[e]);
                            bv[2 * e] = f.x;
                            bv[2 * e + 1] = f.y;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int n = 8 * cc + e;
                            const float an = A2s[n];
                            if (safe) {
                                const float b1 = bv[e] * ex2(an * (MI - Dti));
                                bt[e] = b1 * T5(n);
                                bv[e] = b1;
                            } else {
                                bt[e] = bv[e] * ex2(an * (RI - Dti));
                            }
                            bw[e] = bt[e] * T3(n);
                        }
                        *reinterpret_cast<float4 *>(bprow + 4 * ((2 * cc) ^ sw)) = make_float4(bv[0], bv[1], bv[2], bv[3]);
                        *reinterpret_cast<float4 *>(bprow + 4 * ((2 * cc + 1) ^ sw)) = make_float4(bv[4], bv[5], bv[6], bv[7]);
                        *reinterpret_cast<uint4 *>(smem + kOffBt + i * 128 + ((16u * cc) ^ rx)) =
                            make_uint4(pack_h2(bt[0], bt[1]), pack_h2(bt[2], bt[3]), pack_h2(bt[4], bt[5]), pack_h2(bt[6], bt[7]));
                        *reinterpret_cast<uint4 *>(smem + kOffBw + i * 128 + ((16u * cc) ^ rx)) =
                            make_uint4(pack_h2(bw[0], bw[1]), pack_h2(bw[2], bw[3]), pack_h2(bw[4], bw[5]), pack_h2(bw[6], bw[7]));
                    }
                }
                // C: C' = C exp(A (Dt_i - M_I)) (fp32, kept for the diagonal group); the C side
                // of everything else is C' T1 = C exp(A (Dt_i - R_{I-1})) <= 1 times a table
                // factor.  (C' T1 is formed before the next factor, never T1 times that factor:
                // C' may be large where the product is not small.)  A group outside the split's
                // range takes C exp(A (Dt_i - R_{I-1})) directly (and its diagonal group later
                // reads C from the tile).
                float cr[64];
                {
                    const unsigned char *row = xt + 2 * kTile + i * 128;
                    const float ref = safe ? MI : Rm1;
                    uint32_t wh[32];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + ((16u * cc) ^ rx));
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = bf2_to_f2(ws[e]);
                            const int n = 8 * cc + 2 * e;
                            cr[n] = f.x * ex2(A2s[n] * (Dti - ref));
                            cr[n + 1] = f.y * ex2(A2s[n + 1] * (Dti - ref));
                        }
                    }
                    auto t1 = [&](int n) -> float { return safe ? T1(n) : 1.f; };
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        wh[e] = pack_h2((cr[2 * e] * t1(2 * e)) * T2(2 * e), (cr[2 * e + 1] * t1(2 * e + 1)) * T2(2 * e + 1));
                    tmem_st32u(tmem + lane_off + kTmCh, wh);
                    // one copy per earlier group J: C exp(A (Dt_i - R_J)) = C' T1 G_J; copies J >= I
                    // of a row are never read (those columns of S are replaced), so they are zeros
                    for (int J = 0; J <= 2 * q; ++J) {
                        const bool use = J <= I - 1;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float g0 = use ? Gt(J, 2 * e) : 0.f, g1 = use ? Gt(J, 2 * e + 1) : 0.f;
                            wh[e] = pack_h2((cr[2 * e] * t1(2 * e)) * g0, (cr[2 * e + 1] * t1(2 * e + 1)) * g1);
                        }
                        tmem_st32u(tmem + lane_off + kTmCp + 32 * J, wh);
                    }
                }
                tmem_st_wait();
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_OPS));

                // (4) the diagonal group: S_ij = sum_n C'_in B'_jn, j <= i (fp32; while the MMAs run)
                float d[16];
                if (safe) {
                    const int sw = I & 1;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float4 *brow = reinterpret_cast<const float4 *>(Bp + (16 * I + jj) * 64);
                        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                        for (int c4 = 0; c4 < 16; ++c4) {
                            const float4 bv = brow[c4 ^ sw];
                            s0 = fmaf(cr[4 * c4], bv.x, s0);
                            s1 = fmaf(cr[4 * c4 + 1], bv.y, s1);
                            s2 = fmaf(cr[4 * c4 + 2], bv.z, s2);
                            s3 = fmaf(cr[4 * c4 + 3], bv.w, s3);
                        }
                        d[jj] = jj <= (i & 15) ? (s0 + s1) + (s2 + s3) : 0.f;
                    }
                } else {
                    float dl[16];
                    diag_group_direct(xt + 2 * kTile + i * 128, rx, Bp, A2s, DtW, i, dl);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) d[jj] = dl[jj];
                }

                // (5) S: the copies' products left of the diagonal group, the diagonal group,
                // zeros right of it -> fp16 over S's first 64 columns (each chunk of 16 written
                // columns lies in columns already read)
                wait_bar(ctl, bar(B_SFULL), kb & 1);
                tc_fence_after();
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    float sv[32];
                    tmem_ld32(tmem + lane_off + kTmS + 32 * k4, sv);
                    tmem_ld_wait();
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float v2[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int j = 32 * k4 + 2 * e + u;
                            const int Jg = j >> 4;
                            v2[u] = Jg < I ? sv[2 * e + u] : (Jg == I ? d[j & 15] : 0.f);
                        }
                        w[e] = pack_h2(v2[0], v2[1]);
                    }
                    tmem_st16(tmem + lane_off + kTmS16 + 16 * k4, w);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S16));

                // (6) epilogue: y = Y (bf16) -> this warp's 32-row buffer -> TMA store
                wait_bar(ctl, bar(B_YFULL), kb & 1);
                tc_fence_after();
                if (lane == 0) bulk_wait_read0();   // this warp's previous store has read its buffer
                __syncwarp();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float yv[32];
                    tmem_ld32(tmem + lane_off + kTmY + 32 * half, yv);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t ow[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            ow[e] = pack_bf2(yv[8 * cc + 2 * e], yv[8 * cc + 2 * e + 1]);
                            bad |= bf2_nonfinite(ow[e]);
                        }
                        *reinterpret_cast<uint4 *>(ybuf + swz(lane, 4 * half + cc)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (c * kBlk + 32 * q < p.T) {
                        tma_store_3d(&tm_y, ybuf_a, h * kP, c * kBlk + 32 * q, bi);
                        bulk_commit();
                    }
                    mbar_arrive(bar(B_EMPTY + st));
                }
            }
            // the final state (state rows): h after the last block's product, which (5) waited for
            if (q < 2 && p.final_state) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float hv[32];
                    tmem_ld32(tmem + lane_off + kTmH + 32 * half, hv);
                    tmem_ld_wait();
                    float *dst = p.final_state + ((int64_t)sq * kN + i) * kP + 32 * half;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + e) = make_float4(hv[e], hv[e + 1], hv[e + 2], hv[e + 3]);
                }
            }
        }
        if (lane == 0) bulk_wait0();
        if (__any_sync(0xffffffffu, bad != 0) && lane == 0) set_status(p.status, SSD_ERR_DEVICE);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// Per-device launch setup, once per device: SM count and the dynamic shared
// memory limit.  Returns the SM count (0 on failure).
int diag_device_setup() {
    constexpr int kMaxDev = 64;
    static int sms[kMaxDev] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (sms[dev] > 0) return sms[dev];
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaFuncSetAttribute(ssd_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess)
            return 0;
        sms[dev] = n;
    }
    return sms[dev];
}

}  // namespace

bool diag_supports(const Problem &p) {
    if (p.a_mode != SSD_A_DIAGONAL || p.io_dtype != SSD_DTYPE_BF16) return false;
    if (p.P != kP || p.N != kN) return false;
    if (p.T > (int64_t)INT32_MAX / 2 || p.b * p.H > (int64_t)INT32_MAX) return false;
    return true;
}

size_t diag_workspace_bytes(const Problem &p) {
    (void)p;
    return kStatusBytes;
}

cudaError_t diag_launch(const Problem &p, void *ws, cudaStream_t s) {
    DiagParams dp;
    dp.dt = p.dt;
    dp.A = p.A;
    dp.D = p.D;
    dp.init = p.init;
    dp.final_state = p.final_state;
    dp.status = static_cast<int *>(ws);
    dp.b = (int)p.b;
    dp.T = (int)p.T;
    dp.H = (int)p.H;
    dp.G = (int)p.G;
    dp.nblk = (int)((p.T + kBlk - 1) / kBlk);
    dp.nseq = (int)(p.b * p.H);
    CUtensorMap mx, mB, mC, my;
    if (!make_map(&mx, p.x, (uint64_t)(p.H * p.P), (uint64_t)p.T, (uint64_t)p.b) ||
        !make_map(&mB, p.B, (uint64_t)(p.G * p.N), (uint64_t)p.T, (uint64_t)p.b) ||
        !make_map(&mC, p.C, (uint64_t)(p.G * p.N), (uint64_t)p.T, (uint64_t)p.b) ||
        !make_map(&my, p.y, (uint64_t)(p.H * p.P), (uint64_t)p.T, (uint64_t)p.b, 32))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (e != cudaSuccess) return e;
    const int sms = diag_device_setup();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = dp.nseq < sms ? dp.nseq : sms;
    record_dominant_start(s);
    ssd_diag_kernel<<<grid, kThreads, kSmemBytes, s>>>(mx, mB, mC, my, dp);
    record_dominant_stop(s);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssd
