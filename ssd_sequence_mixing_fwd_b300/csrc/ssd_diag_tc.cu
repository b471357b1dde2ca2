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
// of group J (R_{-1} = 0).  Every product is split at a reference point between
// its two tokens, so that each factor carried by a tensor-core operand is <= 1
// (fp16 operands, fp32 accumulation):
//
//  * S_ij, j in group J < group I of i: exp(A (Dt_i - R_J)) on the C side and
//    exp(A (R_J - Dt_j)) on the B side.  The C side depends on J, so every row
//    keeps one copy of its decayed C per earlier group -- written to TMEM, where
//    the MMA takes it as its A operand -- and the seven products
//    copy_J (128 x 64) x B~_J^T (64 x 16) fill S's columns group by group.
//  * S_ij, j and i in the same group: on the CUDA cores in fp32, split at the
//    group's start R_{I-1} (the B side carries factors up to exp(|A| x the group's
//    Dt range); a group whose factors could leave fp32 takes one exponential per
//    (i, j, n) instead).
//  * h_prev enters through C o exp(A Dt_i) (in TMEM) x h_prev (fp16, shared memory);
//    the state's own product B o w (w <= 1) accumulates onto exp(A Dt_end) o h_prev,
//    which the rows of the state rescale in place in TMEM.
//
// The same map as the chunked algorithm of the other paths (equal up to
// rounding); the block of 128 tokens plays the chunk's part whatever Q is.
//
// One CTA per (batch row, head) at a time (persistent over sequences), 10 warps:
//   warp 0      producer: X, B, C tiles of a block by TMA, its dt by plain loads (two stages)
//   warp 1      TMEM owner; lane 0 issues every MMA
//   warps 2-9   math, two per TMEM lane quarter: thread = TMEM lane = row i of the
//               block (warp w owns lanes 32 (w mod 4) ...), the two warps of a quarter
//               splitting the state dimension n (and the head dim p) in halves; rows
//               0-63 also own the state rows n = i.
// TMEM (512 columns): S 0-127 (fp32), C copies 128-351 (7 x 32, fp16 pairs; S in
// fp16 then takes 128-191), C o exp(A Dt) 352-383, Y 384-447, h 448-511 (lanes 0-63).
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
constexpr int kThreads = 320;      // 10 warps
constexpr int kMathWarps = 8;
constexpr int kTile = 128 * 128;   // 128 rows x 64 16-bit values

// shared memory (byte offsets from a 1024-aligned base)
constexpr int kStageBytes = 3 * kTile;                 // X, B, C (bf16 as loaded; X then fp16)
constexpr int kOffStage = 0;                           // [2 stages]
constexpr int kOffBt = 2 * kStageBytes;                // B~ (fp16, [j][n], 128B swizzle)
constexpr int kOffBw = kOffBt + kTile;                 // B o w (fp16, [j][n])
constexpr int kOffBp = kOffBw + kTile;                 // B' (fp32, [j][64], row-swizzled 16-byte chunks)
constexpr int kOffHp = kOffBp + 2 * kTile;             // h_prev (fp16, [n][p])
constexpr int kOffY = kOffHp + 64 * 128;               // y: [4 quarters][32 rows][128 B]
constexpr int kTabRow = 36;                            // floats per table row (32 + bank padding)
constexpr int kTabRows = 20;                           // per warp: T2 T3 g x 2 groups, G x 2 groups x 7
constexpr int kTabWarpBytes = kTabRows * kTabRow * 4;
constexpr int kOffTab = kOffY + kTile;                 // per math warp: tables of its n half
// The partial diagonal-group sums of the two warps of a quarter ([2][32 rows][16]) share the
// quarter's y buffer: they are read before the buffer takes y.
constexpr int kOffDtW = kOffTab + kMathWarps * kTabWarpBytes;   // per math warp: Dt of all 128 rows
constexpr int kOffA2 = kOffDtW + kMathWarps * 512;     // per math warp: A (log2 units) of its n half
constexpr int kOffDt = kOffA2 + kMathWarps * 128;      // [2 stages][128] dt of the stage's block
constexpr int kOffMisc = kOffDt + 2 * 512;             // TMEM base, abort flag
constexpr int kOffBar = kOffMisc + 16;
constexpr int kNumBars = 8;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

constexpr int B_FULL = 0;     // [2] TMA landed a stage
constexpr int B_EMPTY = 2;    // [2] the math warps are done with a stage (8 warps)
constexpr int B_OPS = 4;      // operands of a block written (8 warps)
constexpr int B_SFULL = 5;    // S, Y_off and the state product are done
constexpr int B_S16 = 6;      // S (fp16) written (8 warps)
constexpr int B_YFULL = 7;    // S X is done

constexpr uint32_t kTmS = 0;
constexpr uint32_t kTmCp = 128;
constexpr uint32_t kTmS16 = 128;
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

// 16-byte chunk c of row r of the B' table sits at chunk c ^ bp_swz(r): eight consecutive
// rows (one warp's stores) spread over all banks, and rows r and r + 16 (the rows two
// halves of a warp read at once) land in different banks.
__device__ __forceinline__ int bp_swz(int r) { return (r ^ (r >> 4)) & 7; }

// The diagonal group of a row whose split factors could leave fp32, over one half of n:
// sum_{n in half} C_in B_jn exp(A_n (Dt_i - Dt_j)) with one exponential per term (C from the
// row's tile, B from the B' table, which holds B itself for such a group).
static __device__ __noinline__ void diag_group_direct(const unsigned char *crow, uint32_t rx, const float *Bp,
                                                      const float *A2h, const float *DtW, int i, int hn,
                                                      float *d) {
    const int I = i >> 4;
    const float Dti = DtW[i];
    float c[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 w = *reinterpret_cast<const uint4 *>(crow + ((16u * (4 * hn + k)) ^ rx));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = bf2_to_f2(ws[e]);
            c[8 * k + 2 * e] = f.x;
            c[8 * k + 2 * e + 1] = f.y;
        }
    }
    for (int jj = 0; jj < 16; ++jj) {
        const int j = 16 * I + jj;
        const float4 *brow = reinterpret_cast<const float4 *>(Bp + j * 64);
        const float dd = Dti - DtW[j];
        float s0 = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
            const float4 bv = brow[(8 * hn + c4) ^ bp_swz(j)];
            const int n = 4 * c4;
            s0 = fmaf(c[n] * bv.x, ex2(A2h[n] * dd), s0);
            s0 = fmaf(c[n + 1] * bv.y, ex2(A2h[n + 1] * dd), s0);
            s0 = fmaf(c[n + 2] * bv.z, ex2(A2h[n + 2] * dd), s0);
            s0 = fmaf(c[n + 3] * bv.w, ex2(A2h[n + 3] * dd), s0);
        }
        d[jj] = jj <= (i & 15) ? s0 : 0.f;
    }
}

__device__ __forceinline__ void pair_sync(int q) { asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory"); }

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
            mbar_init(bar(B_EMPTY + s), kMathWarps);
        }
        mbar_init(bar(B_OPS), kMathWarps);
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_S16), kMathWarps);
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
        // ------------------------------------------------------------ producer
        // The whole warp loads the block's dt (one strided word per token) into the stage; lane 0
        // then arms the stage's barrier (its arrival releases those stores) and issues the TMA.
        int kb = 0;
        bool ok = true;
        for (int sq = blockIdx.x; sq < p.nseq && ok; sq += gridDim.x) {
            const int bi = sq / p.H, h = sq - bi * p.H, g = h / hpg;
            for (int c = 0; c < p.nblk; ++c, ++kb) {
                const int st = kb & 1;
                if (kb >= 2 && !(ok = __all_sync(0xffffffffu, wait_bar(ctl, bar(B_EMPTY + st), ((kb >> 1) - 1) & 1))))
                    break;
                float *dts = reinterpret_cast<float *>(smem + kOffDt + st * 512);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int t = c * kBlk + 32 * m + lane;
                    dts[32 * m + lane] = t < p.T ? __ldg(p.dt + ((int64_t)bi * p.T + t) * p.H + h) : 0.f;
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t dst = sbase + kOffStage + st * kStageBytes;
                    mbar_expect_tx(bar(B_FULL + st), 3 * kTile);
                    tma_load_3d(dst, &tm_x, bar(B_FULL + st), h * kP, c * kBlk, bi);
                    tma_load_3d(dst + kTile, &tm_B, bar(B_FULL + st), g * kN, c * kBlk, bi);
                    tma_load_3d(dst + 2 * kTile, &tm_C, bar(B_FULL + st), g * kN, c * kBlk, bi);
                }
            }
        }
        // after an abort: wait (bounded) for the loads still in flight
        if (!ok && lane == 0)
            for (int k2 = kb - 2; k2 < kb; ++k2)
                if (k2 >= 0) drain_bar(bar(B_FULL + (k2 & 1)), (k2 >> 1) & 1);
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
        const int hn = (warp - 2) >> 2;             // which half of n (and of p) this warp takes
        const int i = 32 * q + lane;                // row of the block (token / state row)
        const int I = i >> 4;                       // 16-row group
        const int lg = (lane >> 4) & 1;             // the group's index within this warp
        const bool need_d = hn == (q < 2 ? 0 : 1);  // this warp's S columns hold the diagonal group
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        float *tab = reinterpret_cast<float *>(smem + kOffTab + (warp - 2) * kTabWarpBytes);
        float *DtW = reinterpret_cast<float *>(smem + kOffDtW + (warp - 2) * 512);
        float *A2h = reinterpret_cast<float *>(smem + kOffA2 + (warp - 2) * 128);
        float *Bp = reinterpret_cast<float *>(smem + kOffBp);
        // partial sums of half hh for this row; 16-byte chunk k at k ^ ((lane >> 1) & 3), so the
        // 64-byte rows of eight consecutive lanes cover all banks
        auto dpart = [&](int hh, int k) {
            return reinterpret_cast<float4 *>(smem + kOffY + q * 4096 + hh * 2048 + lane * 64) + (k ^ ((lane >> 1) & 3));
        };
        unsigned char *ybuf = smem + kOffY + q * 4096;
        const uint32_t ybuf_a = sbase + kOffY + q * 4096;
        // Per-warp tables over this warp's half of n, each factor in (0, 1]:
        //   T2 = exp(A R_{I-1}), T3 = exp(A (Dt_end - R_I)), g = exp(A (R_I - R_{I-1})) for the
        //   warp's two groups, and G_J = exp(A (R_{I-1} - R_J)) for every earlier group J.
        // g multiplies a factor up to exp(|A| (R_I - R_{I-1})) and is at least 2^-110 in a
        // group within the split's range, so no product underflows unless its exact value is
        // below fp32's normal range.
        auto T2 = [&](int k) { return reinterpret_cast<const float4 *>(tab + (0 + lg) * kTabRow)[k >> 2]; };
        auto T3 = [&](int k) { return reinterpret_cast<const float4 *>(tab + (2 + lg) * kTabRow)[k >> 2]; };
        auto Tg = [&](int k) { return reinterpret_cast<const float4 *>(tab + (4 + lg) * kTabRow)[k >> 2]; };
        auto Gt = [&](int J, int k) { return reinterpret_cast<const float4 *>(tab + (6 + 7 * lg + J) * kTabRow)[k >> 2]; };
        auto A4 = [&](int k) { return reinterpret_cast<const float4 *>(A2h)[k >> 2]; };
        uint32_t bad = 0;
        int kb = 0;
        for (int sq = blockIdx.x; sq < p.nseq; sq += gridDim.x) {
            const int bi = sq / p.H, h = sq - bi * p.H;
            __syncwarp();
            const float an_own = p.A[(int64_t)h * kN + 32 * hn + lane] * kLog2e;   // n = 32 hn + lane
            A2h[lane] = an_own;
            float amax = fabsf(an_own);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            // the split's range check uses |A| over all n (the other half from the other warp's values)
            const float amax_other = fabsf(p.A[(int64_t)h * kN + 32 * (1 - hn) + lane]) * kLog2e;
            float am2 = amax_other;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) am2 = fmaxf(am2, __shfl_xor_sync(0xffffffffu, am2, o));
            amax = fmaxf(amax, am2);
            const float a_row = q < 2 ? p.A[(int64_t)h * kN + i] * kLog2e : 0.f;   // state row n = i
            const float Dh = p.D ? p.D[h] : 0.f;
            __syncwarp();
            // the initial state into TMEM (state rows 0-63: quarters 0 and 1; this warp's half of p)
            if (q < 2) {
                float v[32];
                const float *src = p.init ? p.init + ((int64_t)sq * kN + i) * kP + 32 * hn : nullptr;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 f = src ? __ldg(reinterpret_cast<const float4 *>(src + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[e] = f.x;
                    v[e + 1] = f.y;
                    v[e + 2] = f.z;
                    v[e + 3] = f.w;
                }
                tmem_st32(tmem + lane_off + kTmH + 32 * hn, v);
                tmem_st_wait();
            }
            // (1) + (2) of a block, run for block c + 1 while block c's S X is in flight:
            // Dt, the inclusive prefix sums of dt over the block (four interleaved 32-row scans;
            // every warp computes all 128 rows), the warp's tables, and the state rows' h_prev
            // (fp16, for (C o e) h_prev) and rescaling h <- exp(A Dt_end) o h in place (the state
            // product of the previous block, which wrote h, and (C o e) h_prev, which read the
            // h_prev tile, have completed)
            float Dti = 0.f, Dend = 0.f, RI = 0.f, Rm1 = 0.f;
            bool safe = true;
            // (the stage of block kb2 has landed: its dt, and the tiles used later)
            auto prep = [&](int kb2) {
                const int st2 = kb2 & 1;
                wait_bar(ctl, bar(B_FULL + st2), (kb2 >> 1) & 1);
                const float *dts = reinterpret_cast<const float *>(smem + kOffDt + st2 * 512);
                float Dv[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) Dv[m] = dts[32 * m + lane];
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
                __syncwarp();
#pragma unroll
                for (int m = 0; m < 4; ++m) DtW[32 * m + lane] = Dv[m];
                __syncwarp();
                Dti = DtW[i];
                Dend = DtW[127];
                RI = DtW[16 * I + 15];
                Rm1 = I > 0 ? DtW[16 * I - 1] : 0.f;
                // pairs inside the group are split at the group's start: factors up to
                // exp2(|A| (R_I - R_{I-1})) on the B side
                safe = amax * (RI - Rm1) <= kSafeLog2;
#pragma unroll
                for (int l2 = 0; l2 < 2; ++l2) {
                    const int I2 = 2 * q + l2;
                    const float r1 = I2 > 0 ? DtW[16 * I2 - 1] : 0.f;
                    const float r2 = DtW[16 * I2 + 15];
                    tab[(0 + l2) * kTabRow + lane] = ex2(an_own * r1);
                    tab[(2 + l2) * kTabRow + lane] = ex2(an_own * (Dend - r2));
                    tab[(4 + l2) * kTabRow + lane] = ex2(an_own * (r2 - r1));
#pragma unroll
                    for (int J = 0; J < 7; ++J)
                        if (J < I2) tab[(6 + 7 * l2 + J) * kTabRow + lane] = ex2(an_own * (r1 - DtW[16 * J + 15]));
                }
                __syncwarp();
                if (q < 2) {
                    const float an = ex2(a_row * Dend);
                    unsigned char *hrow = smem + kOffHp + i * 128;
                    const uint32_t rxh = (uint32_t)(i & 7) * 16u;
                    float hv[32];
                    tmem_ld32(tmem + lane_off + kTmH + 32 * hn, hv);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int e = 8 * cc;
                        *reinterpret_cast<uint4 *>(hrow + ((16u * (4 * hn + cc)) ^ rxh)) =
                            make_uint4(pack_h2(hv[e], hv[e + 1]), pack_h2(hv[e + 2], hv[e + 3]),
                                       pack_h2(hv[e + 4], hv[e + 5]), pack_h2(hv[e + 6], hv[e + 7]));
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) hv[e] *= an;
                    tmem_st32(tmem + lane_off + kTmH + 32 * hn, hv);
                }
            };
            prep(kb);
            for (int c = 0; c < p.nblk; ++c, ++kb) {
                const int st = kb & 1;

                // (3) operands of row i, this warp's half of n (16-byte chunks 4 hn .. 4 hn + 3)
                wait_bar(ctl, bar(B_FULL + st), (kb >> 1) & 1);
                unsigned char *xt = smem + kOffStage + st * kStageBytes;
                const uint32_t rx = (uint32_t)(i & 7) * 16u;
                {
                    // X: bf16 -> fp16 in place; D x into Y's columns (Y_off accumulates onto it)
                    unsigned char *row = xt + i * 128;
                    uint4 u[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) u[k] = *reinterpret_cast<const uint4 *>(row + ((16u * (4 * hn + k)) ^ rx));
                    if (p.D) {
                        float dx[32];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t ws[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = bf2_to_f2(ws[e]);
                                dx[8 * k + 2 * e] = Dh * f.x;
                                dx[8 * k + 2 * e + 1] = Dh * f.y;
                            }
                        }
                        tmem_st32(tmem + lane_off + kTmY + 32 * hn, dx);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        u[k].x = bf2_to_h2(u[k].x);
                        u[k].y = bf2_to_h2(u[k].y);
                        u[k].z = bf2_to_h2(u[k].z);
                        u[k].w = bf2_to_h2(u[k].w);
                        *reinterpret_cast<uint4 *>(row + ((16u * (4 * hn + k)) ^ rx)) = u[k];
                    }
                }
                {
                    // B: B' = B exp(A (R_{I-1} - Dt_i)) (fp32, for the diagonal group), B~ = B' g =
                    // B exp(A (R_I - Dt_i)), B o w = B~ T3 = B exp(A (Dt_end - Dt_i)) (fp16); a group
                    // outside the split's range keeps B itself in B' and forms B~ directly
                    const unsigned char *row = xt + kTile + i * 128;
                    float *bprow = Bp + i * 64;
                    const int bsw = bp_swz(i);
                    const float bref = safe ? Rm1 : RI;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int cc = 4 * hn + k;
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
                        for (int h4 = 0; h4 < 2; ++h4) {
                            const int k0 = 8 * k + 4 * h4;       // n - 32 hn
                            const float4 a4 = A4(k0), g4 = Tg(k0), t4 = T3(k0);
                            const float av[4] = {a4.x, a4.y, a4.z, a4.w}, gv[4] = {g4.x, g4.y, g4.z, g4.w},
                                        tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int m = 4 * h4 + e;
                                const float b1 = bv[m] * ex2(av[e] * (bref - Dti));
                                bt[m] = safe ? b1 * gv[e] : b1;
                                bw[m] = bt[m] * tv[e];
                                if (safe) bv[m] = b1;
                            }
                        }
                        *reinterpret_cast<float4 *>(bprow + 4 * ((2 * cc) ^ bsw)) = make_float4(bv[0], bv[1], bv[2], bv[3]);
                        *reinterpret_cast<float4 *>(bprow + 4 * ((2 * cc + 1) ^ bsw)) = make_float4(bv[4], bv[5], bv[6], bv[7]);
                        *reinterpret_cast<uint4 *>(smem + kOffBt + i * 128 + ((16u * cc) ^ rx)) =
                            make_uint4(pack_h2(bt[0], bt[1]), pack_h2(bt[2], bt[3]), pack_h2(bt[4], bt[5]), pack_h2(bt[6], bt[7]));
                        *reinterpret_cast<uint4 *>(smem + kOffBw + i * 128 + ((16u * cc) ^ rx)) =
                            make_uint4(pack_h2(bw[0], bw[1]), pack_h2(bw[2], bw[3]), pack_h2(bw[4], bw[5]), pack_h2(bw[6], bw[7]));
                    }
                }
                // C: C~ = C exp(A (Dt_i - R_{I-1})) <= 1 (at least 2^-110 x C in a group within the
                // split's range): the diagonal group's C side as it is, the C side of everything
                // else times a table factor
                float cr[32];
                {
                    const unsigned char *row = xt + 2 * kTile + i * 128;
                    uint32_t wh[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(row + ((16u * (4 * hn + k)) ^ rx));
                        const float4 a4a = A4(8 * k), a4b = A4(8 * k + 4);
                        const float av[8] = {a4a.x, a4a.y, a4a.z, a4a.w, a4b.x, a4b.y, a4b.z, a4b.w};
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = bf2_to_f2(ws[e]);
                            const int m = 8 * k + 2 * e;
                            cr[m] = f.x * ex2(av[2 * e] * (Dti - Rm1));
                            cr[m + 1] = f.y * ex2(av[2 * e + 1] * (Dti - Rm1));
                        }
                    }
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4) {
                        const float4 t = T2(4 * k4);
                        wh[2 * k4] = pack_h2(cr[4 * k4] * t.x, cr[4 * k4 + 1] * t.y);
                        wh[2 * k4 + 1] = pack_h2(cr[4 * k4 + 2] * t.z, cr[4 * k4 + 3] * t.w);
                    }
                    tmem_st16(tmem + lane_off + kTmCh + 16 * hn, wh);
                    // one copy per earlier group J: C exp(A (Dt_i - R_J)) = C~ G_J; copies J >= I
                    // of a row are never read (those columns of S are replaced): zeros
                    for (int J = 0; J <= 2 * q; ++J) {
                        const float z = J <= I - 1 ? 1.f : 0.f;
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            const float4 t = Gt(J, 4 * k4);
                            wh[2 * k4] = pack_h2(cr[4 * k4] * (t.x * z), cr[4 * k4 + 1] * (t.y * z));
                            wh[2 * k4 + 1] = pack_h2(cr[4 * k4 + 2] * (t.z * z), cr[4 * k4 + 3] * (t.w * z));
                        }
                        tmem_st16(tmem + lane_off + kTmCp + 32 * J + 16 * hn, wh);
                    }
                }
                tmem_st_wait();
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_OPS));

                // (4) the diagonal group over this warp's half of n: S_ij = sum_n C~_in B'_jn,
                // j <= i (fp32; while the MMAs run).  The B' rows of the group were written by this
                // warp and its partner: the pair barrier orders them before their use (and the
                // quarter's previous y store has read the buffer the partial sums go to).
                if (hn == 0 && lane == 0) bulk_wait_read0();
                pair_sync(q);
                float d[16];
                if (safe) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j0 = 16 * I + jj;
                        const float4 *b0 = reinterpret_cast<const float4 *>(Bp + j0 * 64);
                        const int s0w = bp_swz(j0) ^ (8 * hn);
                        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 v0 = b0[c4 ^ s0w];
                            s0 = fmaf(cr[4 * c4], v0.x, s0);
                            s1 = fmaf(cr[4 * c4 + 1], v0.y, s1);
                            s2 = fmaf(cr[4 * c4 + 2], v0.z, s2);
                            s3 = fmaf(cr[4 * c4 + 3], v0.w, s3);
                        }
                        d[jj] = jj <= (i & 15) ? (s0 + s1) + (s2 + s3) : 0.f;
                    }
                } else {
                    float dl[16];
                    diag_group_direct(xt + 2 * kTile + i * 128, rx, Bp, A2h, DtW, i, hn, dl);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) d[jj] = dl[jj];
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) *dpart(hn, k) = make_float4(d[4 * k], d[4 * k + 1], d[4 * k + 2], d[4 * k + 3]);
                pair_sync(q);

                // (5) S: the copies' products left of the diagonal group, the diagonal group,
                // zeros right of it -> fp16 (this warp: S columns 64 hn .. 64 hn + 63)
                wait_bar(ctl, bar(B_SFULL), kb & 1);
                tc_fence_after();
                float dsum[16];
                if (need_d) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 a = *dpart(0, k), b = *dpart(1, k);
                        dsum[4 * k] = a.x + b.x;
                        dsum[4 * k + 1] = a.y + b.y;
                        dsum[4 * k + 2] = a.z + b.z;
                        dsum[4 * k + 3] = a.w + b.w;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) dsum[k] = 0.f;
                }
#pragma unroll 1
                for (int k2 = 0; k2 < 2; ++k2) {
                    float sv[32];
                    tmem_ld32(tmem + lane_off + kTmS + 64 * hn + 32 * k2, sv);
                    tmem_ld_wait();
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float v2[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int col = 32 * k2 + 2 * e + u;          // within this warp's 64 columns
                            const int Jg = 4 * hn + (col >> 4);
                            v2[u] = Jg < I ? sv[2 * e + u] : (Jg == I ? dsum[col & 15] : 0.f);
                        }
                        w[e] = pack_h2(v2[0], v2[1]);
                    }
                    tmem_st16(tmem + lane_off + kTmS16 + 32 * hn + 16 * k2, w);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S16));
                if (c + 1 < p.nblk) prep(kb + 1);

                // (6) epilogue: y = Y (bf16; this warp: columns 32 hn ..) -> the quarter's 32-row
                // buffer -> TMA store
                wait_bar(ctl, bar(B_YFULL), kb & 1);
                tc_fence_after();
                pair_sync(q);   // the partial sums in the y buffer have been read
                {
                    float yv[32];
                    tmem_ld32(tmem + lane_off + kTmY + 32 * hn, yv);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t ow[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            ow[e] = pack_bf2(yv[8 * cc + 2 * e], yv[8 * cc + 2 * e + 1]);
                            bad |= bf2_nonfinite(ow[e]);
                        }
                        *reinterpret_cast<uint4 *>(ybuf + swz(lane, 4 * hn + cc)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                pair_sync(q);
                if (lane == 0) {
                    if (hn == 0 && c * kBlk + 32 * q < p.T) {
                        tma_store_3d(&tm_y, ybuf_a, h * kP, c * kBlk + 32 * q, bi);
                        bulk_commit();
                    }
                    mbar_arrive(bar(B_EMPTY + st));
                }
            }
            // the final state (state rows, this warp's half of p): h after the last block's
            // product, which (5) waited for
            if (q < 2 && p.final_state) {
                float hv[32];
                tmem_ld32(tmem + lane_off + kTmH + 32 * hn, hv);
                tmem_ld_wait();
                float *dst = p.final_state + ((int64_t)sq * kN + i) * kP + 32 * hn;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(hv[e], hv[e + 1], hv[e + 2], hv[e + 3]);
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
