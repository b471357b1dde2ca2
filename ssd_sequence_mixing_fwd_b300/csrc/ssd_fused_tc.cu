// ssd_fused_tc.cu -- fused tcgen05/TMA path of the SSD chunked scan (sm_103a).
//
// One persistent kernel evaluates the whole forward pass (Structured State
// Space Duality, "The chunked algorithm takes both"):
//
//   work item = (batch row, 128-token block, k heads of one B/C group)
//     C_blk B_blk^T              once per item, tcgen05 -> TMEM (fp32)
//     per head:
//       cum_i                    prefix sums of dt*A over the block (fp32)
//       S = C B^T o L            L_ij = exp(cum_i - cum_j), j <= i; fp16, kept in TMEM
//       Y_diag = S X             tcgen05, A operand from TMEM
//       s = B^T (w o X)          w_j = exp(cum_end - cum_j); the block's input projection
//       h_prev                   state entering the block, from the previous block's item
//       h = exp(cum_end) h_prev + s        fp32, published for the next block
//       Y_off = C h_prev         tcgen05
//       y = Y_diag + exp(cum_i) Y_off + D x
//
// A chunk of Q = 256 tokens is evaluated as two 128-token blocks: its diagonal
// block is itself split by the chunked algorithm, whose result equals the
// recurrence for any block length, so only rounding differs from a single
// 256-token block.
//
// The serial part -- one state step per block -- runs through an fp32 ring of
// two state slots per (batch, head) in global memory (L2 resident) with one
// release/acquire flag per 32 state rows: the warp that owns rows n..n+31 of a
// head publishes them and the same warp quarter of the next block's item
// waits for exactly those rows.  Items are handed out in block-major order by
// an atomic ticket, so every item that is waited on already runs on a
// resident CTA.  Every wait is bounded: a chain wait that runs out records
// SSD_ERR_TIMEOUT and continues with a zero state; an mbarrier wait that runs
// out records SSD_ERR_TIMEOUT and the CTA winds down.
//
// Precision: C, B and X enter the tensor cores as fp16 (converted in shared
// memory from bf16; exact in the normal range), the masked matrix S, w o X and
// h_prev are rounded to fp16, all accumulation, decay sums and the state are
// fp32 ("When it breaks").
//
// Warp roles (384 threads): warp 0 issues TMA loads and hands out items;
// warp 1 owns TMEM and issues each item's C B^T; warps 2-5 and 6-9 are two
// math groups that take alternate heads (conversion, masks, state step,
// epilogue, TMA stores of y); warp 10 + g issues math group g's tcgen05.mma
// products and publishes its states.
#include <cstring>
#include <mutex>

#include "ssd_ptx.cuh"

namespace ssd {
namespace {

using namespace ptx;

constexpr int kBlk = 128;          // tokens per block = MMA M
constexpr int kP = 64;             // head dim handled by this path
constexpr int kN = 128;            // state rows per MMA tile; N = 128 * NS with NS = 1 or 2
constexpr int kThreads = 384;        // 12 warps: TMA, MMA, 2 x 4 math, 2 publishers
constexpr int kMaxK = 8;           // heads per work item at most

// ---- shared memory map (offsets from a 1024-byte aligned base) -----------
// A C/B stage holds 2 NS boxes of C then 2 NS boxes of B (NS = N / 128): 64 KB or 128 KB;
// two stages for N = 128, one for N = 256 (128 KB either way).
constexpr int kOffStage = 0;                        // 2 stages
constexpr int kOffGroup = 8 * kBox;                 // per math group: X, W (N = 256: group 1's space holds h_prev)
constexpr int kGroupBytes = 2 * kBox;
constexpr int kOffCum = kOffGroup + 2 * kGroupBytes;        // float [2 stages][kMaxK][128]: cum of each head
constexpr int kOffV = kOffCum + 2 * kMaxK * 128 * 4;        // float [2][4][128]
constexpr int kOffDt = kOffV + 2 * 4 * 128 * 4;             // float [2 stages][128][kMaxK]: dt tile
constexpr int kOffItem = kOffDt + 2 * 128 * kMaxK * 4;      // int [2]
constexpr int kOffMisc = kOffItem + 2 * 4;                  // tmem base, abort
constexpr int kOffPub = kOffMisc + 16;                      // int [2][2]: (stream, block) mailbox
constexpr int kOffAD = kOffPub + 16;                        // float [2 stages][kMaxK][2]: A (log2 units), D
constexpr int kOffBar = ((kOffAD + 2 * 2 * kMaxK * 4 + 7) / 8) * 8;  // mbarriers
constexpr int kNumBars = 32;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;   // + alignment slack

// mbarrier indices
constexpr int B_CB_FULL = 0;        // [2] TMA landed C/B of a stage (+ item id)
constexpr int B_CB_CONV = 2;        // [2] C/B converted to fp16 (the 4 warps of one group)
constexpr int B_CB_EMPTY = 4;       // [2] all MMAs reading the stage are done (one arrival per group)
constexpr int B_CBMMA_FULL = 6;     // C B^T of the current item is in TMEM
constexpr int B_CBTMEM_EMPTY = 7;   // every mask of the item has read C B^T (8 warps)
constexpr int B_X_FULL = 8;         // [2] TMA landed X of a head
constexpr int B_X_EMPTY = 10;       // [2] y store has read the X buffer
constexpr int B_XW_READY = 12;      // [2] X converted, w o X written (4 warps)
constexpr int B_S_READY = 14;       // [2] S written to TMEM (4 warps)
constexpr int B_ACC_FULL = 16;      // [2] Y_diag and s are in TMEM
constexpr int B_HP_READY = 18;      // [2] h_prev (fp16) written, s read (4 warps)
constexpr int B_YO_FULL = 20;       // [2] Y_off is in TMEM
constexpr int B_CUM_READY = 22;     // [2] cum of every head of the stage's item is in shared memory
constexpr int B_PUB_FULL = 24;      // [2] a group stored a state: publish it (4 warps)
constexpr int B_PUB_DONE = 26;      // [2] the publisher has taken the mailbox
constexpr int B_W_FREE = 28;        // [2] the previous y store has read the W buffer (leader)
constexpr int B_Y_READY = 30;       // [2] all rows of y are in the W buffer (4 warps)

// TMEM columns (512 allocated)
constexpr uint32_t kTmCB = 0;                       // 128 cols: C B^T (fp32)
__host__ __device__ constexpr uint32_t tm_S(int g) { return 128 + 192 * g; }     // 64 cols: S (fp16 pairs); N = 128: then Y_off
__host__ __device__ constexpr uint32_t tm_Yd(int g) { return 192 + 192 * g; }    // 64 cols
__host__ __device__ constexpr uint32_t tm_Acc(int g) { return 256 + 192 * g; }   // 64 cols: s (N = 256: 128 cols, then Y_off)

struct FusedParams {
    const float *dt, *A, *D, *init;
    float *final_state;
    float *ring;          // (b*H, 2, N, P)
    unsigned *flags;      // (b*H, 2, 4)
    int *status;
    unsigned *ticket;
    int b, T, H, G, k, HG, nblk, total_items;
    int dt_tma;           // dt tile comes by TMA (k and H multiples of 4), else by thread loads
    int64_t chain_spin;
    int64_t withhold;
};

__device__ __forceinline__ void decode_item(const FusedParams &p, int t, int &bi, int &blk, int &hgi) {
    const int per = p.b * p.HG;
    blk = t / per;
    const int rem = t - blk * per;
    bi = rem / p.HG;
    hgi = rem - bi * p.HG;
}

// C and B of a stage, bf16 -> fp16 in place: row r of each of the nbox boxes.  Chunk
// c ^ (r & 7): eight consecutive rows touch eight different 16-byte bank groups (walking
// chunk c of every row would put a quarter warp on the same four banks).
__device__ __noinline__ void convert_stage_rows(unsigned char *base, int nbox, int r) {
    const uint32_t rx = (uint32_t)(r & 7) * 16u;
#pragma unroll 1
    for (int bx = 0; bx < nbox; ++bx) {
        unsigned char *row = base + bx * kBox + r * 128;
        uint4 u[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) u[c] = *reinterpret_cast<const uint4 *>(row + ((16u * c) ^ rx));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            u[c].x = bf2_to_h2(u[c].x);
            u[c].y = bf2_to_h2(u[c].y);
            u[c].z = bf2_to_h2(u[c].z);
            u[c].w = bf2_to_h2(u[c].w);
            *reinterpret_cast<uint4 *>(row + ((16u * c) ^ rx)) = u[c];
        }
    }
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                     const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y,
                     const __grid_constant__ CUtensorMap tm_dt, const FusedParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // N = 128 NS state rows.  N = 128: two math groups, two C/B stages.  N = 256: one math
    // group (its TMEM takes two 64-column state accumulators), one C/B stage, and the
    // other group's buffers hold the 256 x 64 fp16 h_prev.
    constexpr int kNr = kN * NS;
    constexpr int NG = (NS == 1) ? 2 : 1;
    constexpr int NST = (NS == 1) ? 2 : 1;
    constexpr int kStage = 4 * NS * kBox;

    float *cumT = reinterpret_cast<float *>(smem + kOffCum);     // [2 stages][kMaxK][128]
    float *vS = reinterpret_cast<float *>(smem + kOffV);         // [2][4][128]
    float *dtT = reinterpret_cast<float *>(smem + kOffDt);       // [2][128][k]
    int *itemS = reinterpret_cast<int *>(smem + kOffItem);       // [2]
    volatile int *pubS = reinterpret_cast<volatile int *>(smem + kOffPub);   // [2][2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
    auto stage_c = [&](int st, int box) -> uint32_t { return sbase + kOffStage + st * kStage + box * kBox; };
    auto stage_b = [&](int st, int box) -> uint32_t {
        return sbase + kOffStage + st * kStage + (2 * NS + box) * kBox;
    };
    auto grp_x = [&](int g) -> uint32_t { return sbase + kOffGroup + g * kGroupBytes; };
    auto grp_w = [&](int g) -> uint32_t { return sbase + kOffGroup + g * kGroupBytes + kBox; };
    // h_prev (fp16, N x 64, MN-major) for C h_prev: the W buffer, or 32 KB of spare buffers
    auto grp_hp = [&](int g) -> uint32_t { return NS == 1 ? grp_w(g) : sbase + kOffGroup + kGroupBytes; };
    const Ctl ctl{p.status, abort_flag};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_CB_FULL + s), 1);
            mbar_init(bar(B_CB_CONV + s), 4);
            mbar_init(bar(B_CB_EMPTY + s), NG);
            mbar_init(bar(B_X_FULL + s), 1);
            mbar_init(bar(B_X_EMPTY + s), 1);
            mbar_init(bar(B_XW_READY + s), 4);
            mbar_init(bar(B_S_READY + s), 4);
            mbar_init(bar(B_ACC_FULL + s), 1);
            mbar_init(bar(B_HP_READY + s), 4);
            mbar_init(bar(B_YO_FULL + s), 1);
            mbar_init(bar(B_CUM_READY + s), 1);
        }
        mbar_init(bar(B_CBMMA_FULL), 1);
        mbar_init(bar(B_CBTMEM_EMPTY), 4 * NG);
        for (int g2 = 0; g2 < 2; ++g2) {
            mbar_init(bar(B_PUB_FULL + g2), 4);
            mbar_init(bar(B_PUB_DONE + g2), 1);
            mbar_init(bar(B_W_FREE + g2), 1);
            mbar_init(bar(B_Y_READY + g2), 4);
        }
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
    const int k = p.k;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0, flat = 0;
            int xcnt[2] = {0, 0};
            int last_cb_use[2] = {-1, -1};
            bool ok = true;
            for (;; ++it) {
                const int st = it % NST;
                if (it >= NST && !(ok = wait_bar(ctl, bar(B_CB_EMPTY + st), ((it / NST) - 1) & 1))) break;
                const unsigned t = atomicAdd(p.ticket, 1u);
                const int id = t < (unsigned)p.total_items ? (int)t : -1;
                itemS[st] = id;
                if (id < 0) {
                    mbar_arrive(bar(B_CB_FULL + st));
                    break;
                }
                int bi, blk, hgi;
                decode_item(p, id, bi, blk, hgi);
                const int t0 = blk * kBlk;
                const int grp = (hgi * k) / (p.H / p.G);
                {
                    float *ad = reinterpret_cast<float *>(smem + kOffAD) + st * (2 * kMaxK);
                    float av[kMaxK], dv[kMaxK];
#pragma unroll
                    for (int jj = 0; jj < kMaxK; ++jj) {
                        av[jj] = jj < k ? p.A[hgi * k + jj] : 0.f;
                        dv[jj] = (jj < k && p.D) ? p.D[hgi * k + jj] : 0.f;
                    }
#pragma unroll
                    for (int jj = 0; jj < kMaxK; ++jj) {
                        ad[2 * jj] = av[jj] * kLog2e;
                        ad[2 * jj + 1] = dv[jj];
                    }
                }
                mbar_expect_tx(bar(B_CB_FULL + st), kStage + (p.dt_tma ? kBlk * k * 4 : 0));
                last_cb_use[st] = it;
                if (p.dt_tma) tma_load_3d(sbase + kOffDt + st * (kBlk * kMaxK * 4), &tm_dt, bar(B_CB_FULL + st),
                                          hgi * k, t0, bi);
                for (int bx = 0; bx < 2 * NS; ++bx) {
                    tma_load_3d(stage_c(st, bx), &tm_C, bar(B_CB_FULL + st), grp * kNr + 64 * bx, t0, bi);
                    tma_load_3d(stage_b(st, bx), &tm_B, bar(B_CB_FULL + st), grp * kNr + 64 * bx, t0, bi);
                }
                for (int j = 0; j < k; ++j, ++flat) {
                    const int g = flat % NG;
                    if (xcnt[g] >= 1 && !(ok = wait_bar(ctl, bar(B_X_EMPTY + g), (xcnt[g] - 1) & 1))) break;
                    mbar_expect_tx(bar(B_X_FULL + g), kBox);
                    tma_load_3d(grp_x(g), &tm_x, bar(B_X_FULL + g), (hgi * k + j) * kP, t0, bi);
                    ++xcnt[g];
                }
                if (!ok) break;
            }
            // After an abort, wait (bounded) until every load issued has landed,
            // so no copy writes shared memory after the CTA has gone.  In a normal
            // finish every load has been consumed already.
            if (!ok) {
                for (int s = 0; s < 2; ++s) {
                    if (last_cb_use[s] >= 0) drain_bar(bar(B_CB_FULL + s), (last_cb_use[s] / NST) & 1);
                    if (xcnt[s] >= 1) drain_bar(bar(B_X_FULL + s), (xcnt[s] - 1) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ prefix sums + C B^T issuer
        // Per item, the whole warp computes cum_t = sum_{u <= t} dt_u A log2(e) of each of
        // the item's heads into shared memory (four interleaved 32-row scans, rows
        // lane + 32 m), so the math groups start a head without a scan.  Lane 0 owns TMEM
        // and issues the item's C B^T once its C and B are fp16 and every mask of the
        // previous item has read the previous C B^T.
        {
            const uint32_t id_cb = idesc_f16(128, 128, 0, 0);
            for (int it = 0;; ++it) {
                const int st = it % NST;
                const uint32_t par = (it / NST) & 1;
                // every lane waits (no lane idles at a shuffle while another waits); a vote
                // keeps the lanes together when a wait gives up
                if (!__all_sync(0xffffffffu, wait_bar(ctl, bar(B_CB_FULL + st), par))) break;
                if (itemS[st] < 0) break;
                if (!p.dt_tma && !__all_sync(0xffffffffu, wait_bar(ctl, bar(B_CB_CONV + st), par))) break;
                {
                    const float *tile = dtT + st * (kBlk * kMaxK);
                    const float *adS = reinterpret_cast<const float *>(smem + kOffAD) + st * (2 * kMaxK);
                    float *ct = cumT + st * (kMaxK * 128);
                    for (int jj = 0; jj < k; ++jj) {
                        // rows lane + 32 m: four interleaved 32-row scans, then the quarter offsets
                        const float Aj = adS[2 * jj];
                        float v[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m) v[m] = tile[(32 * m + lane) * k + jj] * Aj;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const float u2 = __shfl_up_sync(0xffffffffu, v[m], o);
                                if (lane >= o) v[m] += u2;
                            }
                        }
                        float run = 0.f;
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            ct[jj * 128 + 32 * m + lane] = run + v[m];
                            run += __shfl_sync(0xffffffffu, v[m], 31);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_CUM_READY + st));
                if (!__all_sync(0xffffffffu, wait_bar(ctl, bar(B_CB_CONV + st), par))) break;
                if (it >= 1 && !__all_sync(0xffffffffu, wait_bar(ctl, bar(B_CBTMEM_EMPTY), (it - 1) & 1))) break;
                if (lane == 0) {
                    tc_fence_after();
                    // K steps of 16: +32 bytes inside a swizzle atom, next atom = next box
                    const uint64_t ca = sdesc(stage_c(st, 0), 16, 1024), cb = sdesc(stage_b(st, 0), 16, 1024);
                    for (int kk = 0; kk < 8 * NS; ++kk) {
                        const uint64_t o = (uint64_t)((kk >> 2) * (kBox >> 4) + 2 * (kk & 3));
                        mma_ss(tmem + kTmCB, ca + o, cb + o, id_cb, kk > 0);
                    }
                    mma_commit(bar(B_CBMMA_FULL));
                }
                __syncwarp();
            }
        }
    } else if (warp >= 10 && warp < 10 + NG) {
        // ------------------------------------------------------------ per-group issuer + publisher
        // Warp 10 + g serves math group g only, so neither group's products wait behind
        // the other's.  An event loop:
        //  * publications: after the group's four warps have stored a block's state
        //    (mbarrier arrive = CTA-scope release), a GPU-scope fence makes those stores
        //    visible and the 32-row counters of the ring slot grow by 32;
        //  * products of the group's current head, each as soon as its inputs are ready:
        //    s = B^T (w o X), then Y_diag (+)= S X (its completion frees the X buffer),
        //    then Y_off = C h_prev (after the item's last one, the stage's C/B are released;
        //    N = 128 writes it into the S columns once S X has completed).
        const int g = warp - 10;
        if (lane == 0) {
            const uint32_t id_st = idesc_f16(128, kP, 1, 1);
            const uint32_t id_yx = idesc_f16(128, kP, 0, 1);
            const bool has_d = p.D != nullptr;
            int n = 0, ph = 0, m = 0;
            int f = g, it = g / k, j = g - (g / k) * k;     // group g's n-th head is flat head NG n + g
            uint32_t idle = 0;
            for (;;) {
                bool progress = false;
                const int st = it % NST;
                if (ph == 0) {
                    if (mbar_test(bar(B_XW_READY + g), n & 1) && mbar_test(bar(B_CB_CONV + st), (it / NST) & 1)) {
                        tc_fence_after();
                        // A = B^T (MN-major, two 64-row atoms), B = w o X (MN-major)
                        // one M = 128 product per 128 state rows (A = two 64-row atoms of B each)
                        const uint64_t db = sdesc(grp_w(g), kBox, 1024);
#pragma unroll
                        for (int hf = 0; hf < NS; ++hf) {
                            const uint64_t da = sdesc(stage_b(st, 2 * hf), kBox, 1024);
                            for (int kk = 0; kk < 8; ++kk)   // K steps of 16 rows: +2048 bytes
                                mma_ss(tmem + tm_Acc(g) + 64 * hf, da + 128 * kk, db + 128 * kk, id_st, kk > 0);
                        }
                        mma_commit(bar(B_ACC_FULL + g));
                        ph = 1;
                        progress = true;
                    }
                } else if (ph == 1) {
                    if (mbar_test(bar(B_S_READY + g), n & 1)) {
                        tc_fence_after();
                        const uint64_t dx = sdesc(grp_x(g), kBox, 1024);
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tmem + tm_Yd(g), tmem + tm_S(g) + 8 * kk, dx + 128 * kk, id_yx, (kk > 0) || has_d);
                        mma_commit(bar(B_X_EMPTY + g));
                        ph = 2;
                        progress = true;
                    }
                } else {
                    // (N = 128: C h_prev writes the S columns, so S X must have completed)
                    if (mbar_test(bar(B_HP_READY + g), n & 1) && (NS == 2 || mbar_test(bar(B_X_EMPTY + g), n & 1))) {
                        tc_fence_after();
                        // A = C (K-major), B = h_prev (MN-major)
                        const uint64_t ca = sdesc(stage_c(st, 0), 16, 1024), db = sdesc(grp_hp(g), kBox, 1024);
                        for (int kk = 0; kk < 8 * NS; ++kk) {
                            const uint64_t o = (uint64_t)((kk >> 2) * (kBox >> 4) + 2 * (kk & 3));
                            mma_ss(tmem + (NS == 1 ? tm_S(g) : tm_Acc(g)), ca + o, db + 128 * kk, id_yx, kk > 0);
                        }
                        mma_commit(bar(B_YO_FULL + g));
                        if (j + NG >= k) mma_commit(bar(B_CB_EMPTY + st));  // the group's last head of the item
                        ph = 0;
                        ++n;
                        f += NG;
                        it = f / k;
                        j = f - it * k;
                        progress = true;
                    }
                }
                if (mbar_test(bar(B_PUB_FULL + g), m & 1)) {
                    const int sidx = pubS[2 * g], bh = pubS[2 * g + 1];
                    if (sidx < 0) break;            // the group has finished every head
                    fence_acq_rel_gpu();
                    // bh = 2 block + half: the four 32-row counters of one 128-row half
                    unsigned *fl = p.flags + ((int64_t)sidx * 2 + ((bh >> 1) & 1)) * 4 * NS + 4 * (bh & 1);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) red_relaxed_add(fl + qq, 32u);
                    mbar_arrive(bar(B_PUB_DONE + g));
                    ++m;
                    progress = true;
                }
                if (progress) {
                    idle = 0;
                } else if (++idle > kIdleSpin) {
                    set_status(p.status, SSD_ERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                } else if ((idle & 1023u) == 0 && *abort_flag) {
                    break;
                }
            }
        }
    } else if (warp >= 2 && warp < 2 + 4 * NG) {
        // ------------------------------------------------------------ math groups
        const int g = (warp - 2) >> 2;
        const int q = warp & 3;                 // TMEM lane quarter
        const int r = 32 * q + lane;            // row of this thread (token or state row)
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const bool leader = (warp == 2 + 4 * g) && lane == 0;
        float *vq = vS + 512 * g;
        // Nonzero once a y value of this thread is not finite.  The matrix operands are fp16
        // (C, B, x, h_prev, and S, which C B^T bounds since every decay factor is <= 1); one of
        // them beyond the fp16 range becomes inf, and an inf operand leaves a non-finite value
        // in some y it multiplies into (inf, or NaN where it meets a zero), so checking y covers
        // every operand: reported at the end as SSD_ERR_DEVICE.
        uint32_t bad = 0;
        unsigned char *xbuf = smem + kOffGroup + g * kGroupBytes;
        unsigned char *wbuf = xbuf + kBox;
        {
            // the column blocks right of this quarter's diagonal block are zero in every S
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
            for (int J = 1; J < 4; ++J)
                if (J > q) tmem_st16(tmem + lane_off + tm_S(g) + 16 * J, z);
            tmem_st_wait();
        }
        int it = 0, flat = 0, hcnt = 0, npub = 0;
        bool ok = true;
        bool conv_ahead = false;                // this warp converted the current stage's rows ahead
        for (;; ++it) {
            const int st = it % NST;
            if (!(ok = wait_bar(ctl, bar(B_CB_FULL + st), (it / NST) & 1))) break;
            const int id = itemS[st];
            if (id < 0) break;
            int bi, blk, hgi;
            decode_item(p, id, bi, blk, hgi);
            const int t0 = blk * kBlk;
            const int L = min(kBlk, p.T - t0);
            const int j0 = (g - flat % NG + NG) % NG;   // first head of this group in the item
            // C and B of this stage: bf16 -> fp16 in place, row r of all four boxes.  The
            // group that owns the item's first head does it: that group has no Y_off
            // of the previous item outstanding, so C B^T of this item never waits on
            // the other group's state chain.
            // (N = 128: a warp that found this stage already landed during its last head of the
            // previous item has converted its rows then, while it waited for C h_prev)
            if (j0 == 0 && !conv_ahead) {
                convert_stage_rows(smem + kOffStage + st * kStage, 4 * NS, r);
                if (!p.dt_tma) {
                    // dt tile by thread loads (rows past the sequence end are zero)
                    float *tile = dtT + st * (kBlk * kMaxK);
                    for (int jj = 0; jj < k; ++jj)
                        tile[r * k + jj] = (r < L) ? p.dt[((int64_t)bi * p.T + t0 + r) * p.H + hgi * k + jj] : 0.f;
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_CB_CONV + st));
            }
            conv_ahead = false;
            const int my_count = (k - j0 + NG - 1) / NG;
            // A (log2 units) and D of the item's heads: written by the producer with the stage
            const float *adS = reinterpret_cast<const float *>(smem + kOffAD) + st * (2 * kMaxK);
            // the prefix sums of the item's heads (warp 1; it reads a thread-loaded dt tile only
            // after the converting group has written it)
            if (my_count > 0 && !(ok = wait_bar(ctl, bar(B_CUM_READY + st), (it / NST) & 1))) break;
            if (my_count == 0) {
                // no head of this item here: nothing of this group reads C B^T or the stage
                if (lane == 0) mbar_arrive(bar(B_CBTMEM_EMPTY));
                if (leader) mbar_arrive(bar(B_CB_EMPTY + st));
            }
            for (int s = 0; s < my_count && ok; ++s) {
                const int j = j0 + NG * s;
                const int h = hgi * k + j;
                const float Dh = adS[2 * j + 1];
                // (1) cum (log2 units) of this head, computed per item by warp 1: own row ci,
                //     the block total, R = cum at row 32q - 1, and the rank-1 factors
                //     v_j = 2^(R - cum_j) of the rows of earlier quarters
                const float *cum = cumT + st * (kMaxK * 128) + j * 128;
                const float ci = cum[r];
                const float total = cum[127];
                const float Rq = q ? cum[32 * q - 1] : 0.f;
#pragma unroll
                for (int m = 0; m < 3; ++m)
                    if (m < q) vq[128 * q + 32 * m + lane] = ex2(Rq - cum[32 * m + lane]);
                __syncwarp();
                // (2) X -> fp16 in place (for S X); w o X -> W; Y_diag <- D x (exact fp32, the
                //     S X products accumulate onto it)
                // the previous head's y store must have read the W buffer before it is reused
                if (leader) {
                    bulk_wait_read0();
                    mbar_arrive(bar(B_W_FREE + g));
                }
                if (!(ok = wait_bar(ctl, bar(B_W_FREE + g), hcnt & 1))) break;
                if (!(ok = wait_bar(ctl, bar(B_X_FULL + g), hcnt & 1))) break;
                {
                    const float w = ex2(total - ci);
                    const float2 w2 = make_float2(w, w), d2 = make_float2(Dh, Dh);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float dx[32];
                        uint4 xin[4];
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc)
                            xin[cc] = *reinterpret_cast<const uint4 *>(xbuf + swz(r, 4 * half + cc));
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const uint32_t off = swz(r, 4 * half + cc);
                            const uint32_t uw[4] = {xin[cc].x, xin[cc].y, xin[cc].z, xin[cc].w};
                            uint32_t xo[4], wo[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = bf2_to_f2(uw[e]);
                                xo[e] = pack_h2f(f);
                                wo[e] = pack_h2f(mul2(f, w2));
                                const float2 dv = mul2(f, d2);
                                dx[8 * cc + 2 * e] = dv.x;
                                dx[8 * cc + 2 * e + 1] = dv.y;
                            }
                            *reinterpret_cast<uint4 *>(xbuf + off) = make_uint4(xo[0], xo[1], xo[2], xo[3]);
                            *reinterpret_cast<uint4 *>(wbuf + off) = make_uint4(wo[0], wo[1], wo[2], wo[3]);
                        }
                        if (p.D) tmem_st32(tmem + lane_off + tm_Yd(g) + 32 * half, dx);
                    }
                    if (p.D) tmem_st_wait();
                    fence_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_XW_READY + g));
                }
                // (3) mask: S_ij = CB_ij * 2^(cum_i - cum_j), j <= i
                //   column block J < q: rank-1 form u_i * v_j around R = cum at row 32q-1
                //   J == q: direct; J > q: zero
                if (s == 0 && !(ok = wait_bar(ctl, bar(B_CBMMA_FULL), it & 1))) break;
                tc_fence_after();
                {
                    const float u = ex2(ci - Rq);
                    const float2 u2 = make_float2(u, u);
                    // column blocks J > q stay zero: written once per CTA before the loop.
                    // (a rolled loop: unrolled over J it made the kernel ~11 KB larger, and
                    // code size, through the instruction cache, costs more than the loop)
#pragma unroll 1
                    for (int J = 0; J <= q; ++J) {
                        uint32_t pk[16];
                        float c[32];
                        tmem_ld32(tmem + lane_off + kTmCB + 32 * J, c);
                        tmem_ld_wait();
                        if (J < q) {
                            const float2 *vv = reinterpret_cast<const float2 *>(vq + 128 * q + 32 * J);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                pk[e] = pack_h2f(mul2(mul2(make_float2(c[2 * e], c[2 * e + 1]), u2), vv[e]));
                        } else {
                            const float *cj = cum + 32 * J;
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float m0 = (e <= lane) ? ex2(ci - cj[e]) : 0.f;
                                const float m1 = (e + 1 <= lane) ? ex2(ci - cj[e + 1]) : 0.f;
                                pk[e >> 1] = pack_h2f(mul2(make_float2(c[e], c[e + 1]), make_float2(m0, m1)));
                            }
                        }
                        tmem_st16(tmem + lane_off + tm_S(g) + 16 * J, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(bar(B_S_READY + g));
                        if (s == my_count - 1) mbar_arrive(bar(B_CBTMEM_EMPTY));
                    }
                }
                // (4) state step: h_prev (fp16) -> W buffer for C h_prev; h = 2^total h_prev + s; publish
                if (!(ok = wait_bar(ctl, bar(B_ACC_FULL + g), hcnt & 1))) break;
                tc_fence_after();
                {
                    const float a = ex2(total);
                    const float2 a2 = make_float2(a, a);
                    const int64_t sidx = (int64_t)bi * p.H + h;
                    const bool first = (blk == 0);
                    const bool last = (blk == p.nblk - 1);
                    unsigned char *hpbuf = smem + (grp_hp(g) - sbase);
                    // one pass per 128 state rows (N = 256: rows r and r + 128 of this thread)
#pragma unroll 1
                    for (int hf = 0; hf < NS; ++hf) {
                    const int nrow = r + 128 * hf;
                    // Ring slots are chunk-major -- float4 chunk e of state row n at
                    // (e * N + n) -- so each warp-wide access is 512 contiguous bytes.
                    // init_state / final_state keep the caller's (N, P) row-major layout.
                    // A slot's counter (one per 32 state rows) grows by 32 per publication.
                    const float4 *src = nullptr;
                    int src_stride = 1;                 // float4 step between chunks of a row
                    if (first) {
                        if (p.init) src = reinterpret_cast<const float4 *>(p.init + (sidx * kNr + nrow) * kP);
                    } else {
                        const int ps = (blk - 1) & 1;
                        const unsigned *fl = p.flags + (sidx * 2 + ps) * 4 * NS + q + 4 * hf;
                        const unsigned want = 32u * (unsigned)((blk - 1) / 2 + 1);
                        bool got = false;
                        for (int64_t i = 0; i < p.chain_spin; ++i) {
                            if (ld_acquire(fl) >= want) {
                                got = true;
                                break;
                            }
                        }
                        if (got) {
                            src = reinterpret_cast<const float4 *>(p.ring + (sidx * 2 + ps) * kNr * kP) + nrow;
                            src_stride = kNr;
                        } else {
                            set_status(p.status, SSD_ERR_TIMEOUT);
                        }
                    }
                    float4 *dst = nullptr;
                    int dst_stride = 1;
                    if (last) {
                        if (p.final_state) dst = reinterpret_cast<float4 *>(p.final_state + (sidx * kNr + nrow) * kP);
                    } else {
                        dst = reinterpret_cast<float4 *>(p.ring + (sidx * 2 + (blk & 1)) * kNr * kP) + nrow;
                        dst_stride = kNr;
                    }
                    float4 hp[16];
                    if (src) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) hp[e] = __ldcg(src + e * src_stride);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) hp[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    uint32_t hk[32];                    // h_prev as fp16 pairs, for C h_prev
                    if constexpr (NS == 1) {
                        // N = 128: C h_prev goes to the S columns (free once S X has completed:
                        // the issuer also waits for that), so it needs h_prev only and is
                        // signalled before s is read and before the global stores, whose
                        // completion the release of this arrive would otherwise wait for
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) {
                            const float4 u0 = hp[2 * cc], u1 = hp[2 * cc + 1];
                            *reinterpret_cast<uint4 *>(hpbuf + swz(nrow, cc)) =
                                make_uint4(pack_h2(u0.x, u0.y), pack_h2(u0.z, u0.w), pack_h2(u1.x, u1.y), pack_h2(u1.z, u1.w));
                        }
                        fence_async_smem();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_HP_READY + g));
                    }
                    // s is read from TMEM while the global loads are in flight
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float sv[32];
                        tmem_ld32(tmem + lane_off + tm_Acc(g) + 64 * hf + 32 * half, sv);
                        tmem_ld_wait();
#pragma unroll
                        for (int e8 = 0; e8 < 8; ++e8) {
                            const int e = 8 * half + e8;
                            const float4 t4 = hp[e];
                            if (dst) {
                                const float2 lo = fma2(a2, make_float2(t4.x, t4.y), make_float2(sv[4 * e8], sv[4 * e8 + 1]));
                                const float2 hi = fma2(a2, make_float2(t4.z, t4.w),
                                                       make_float2(sv[4 * e8 + 2], sv[4 * e8 + 3]));
                                __stcg(dst + e * dst_stride, make_float4(lo.x, lo.y, hi.x, hi.y));
                            }
                            if constexpr (NS == 2) {
                                hk[2 * e] = pack_h2(t4.x, t4.y);
                                hk[2 * e + 1] = pack_h2(t4.z, t4.w);
                            }
                        }
                    }
                    if constexpr (NS == 2) {
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
                            *reinterpret_cast<uint4 *>(hpbuf + swz(nrow, cc)) =
                                make_uint4(hk[4 * cc], hk[4 * cc + 1], hk[4 * cc + 2], hk[4 * cc + 3]);
                        // N = 256 (chain-bound): each warp publishes its own 32 rows of each half
                        // as soon as they are stored -- every lane fences its stores at GPU
                        // scope, then one lane bumps the quarter's counter -- so the next block's
                        // warp of the same quarter waits neither for the other warps nor for
                        // this block's second half
                        if (!last && (int64_t)blk != p.withhold) {
                            fence_acq_rel_gpu();
                            __syncwarp();
                            if (lane == 0)
                                red_relaxed_add(p.flags + (sidx * 2 + (blk & 1)) * 4 * NS + q + 4 * hf, 32u);
                        }
                    }
                    }
                    if constexpr (NS == 2) {
                        fence_async_smem();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_HP_READY + g));
                    }
                    if (NS == 1 && !last && (int64_t)blk != p.withhold) {
                        // Hand the publication to this group's issuer warp, which makes the
                        // stores visible at GPU scope (fence) and bumps the counters, so these
                        // warps do not wait for the fence.  (h_prev is signalled first: the
                        // issuer starts C h_prev before it fences.)
                        if (leader) {
                            // (a wait that runs out has set the status and the abort flag; the
                            // other waits then end quickly)
                            if (npub >= 1) wait_bar(ctl, bar(B_PUB_DONE + g), (npub - 1) & 1);
                            pubS[2 * g] = (int)sidx;
                            pubS[2 * g + 1] = 2 * blk + (NS - 1);   // N = 256: the second half
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_PUB_FULL + g));
                        ++npub;
                    }

                }
                // N = 128: in the group's last head of the item, while C h_prev runs, convert the
                // next item's C/B if this group owns that item's first head and its tiles have
                // landed (a non-blocking test; otherwise the conversion waits for the item start)
                if constexpr (NS == 1) {
                    if (s == my_count - 1 && p.dt_tma && (flat + k) % NG == g) {
                        const int st2 = (it + 1) % NST;
                        const bool landed = __shfl_sync(0xffffffffu,
                                                        lane == 0 ? (int)mbar_test(bar(B_CB_FULL + st2), ((it + 1) / NST) & 1) : 0, 0);
                        if (landed && itemS[st2] >= 0) {
                            convert_stage_rows(smem + kOffStage + st2 * kStage, 4 * NS, r);
                            fence_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar(B_CB_CONV + st2));
                            conv_ahead = true;
                        }
                    }
                }
                // (5) epilogue: y = Y_diag + 2^cum_i Y_off + D x  ->  bf16 into the W buffer, TMA store
                if (!(ok = wait_bar(ctl, bar(B_YO_FULL + g), hcnt & 1))) break;
                tc_fence_after();
                {
                    const float gi = ex2(ci);
                    const float2 g2 = make_float2(gi, gi);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float yd[32], yo[32];
                        tmem_ld32(tmem + lane_off + tm_Yd(g) + 32 * half, yd);
                        tmem_ld32(tmem + lane_off + (NS == 1 ? tm_S(g) : tm_Acc(g)) + 32 * half, yo);
                        tmem_ld_wait();
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            uint32_t ow[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c0 = 8 * cc + 2 * e;
                                const float2 yv = fma2(g2, make_float2(yo[c0], yo[c0 + 1]),
                                                       make_float2(yd[c0], yd[c0 + 1]));
                                ow[e] = pack_bf2(yv.x, yv.y);
                                bad |= bf2_nonfinite(ow[e]);
                            }
                            *reinterpret_cast<uint4 *>(wbuf + swz(r, 4 * half + cc)) =
                                make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        }
                    }
                    if constexpr (NS == 1) {
                        // C h_prev overwrote the zero blocks right of this quarter's diagonal:
                        // restore them for the next head's S
                        uint32_t z[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
                        for (int J = 1; J < 4; ++J)
                            if (J > q) tmem_st16(tmem + lane_off + tm_S(g) + 16 * J, z);
                    }
                    tc_fence_before();
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_Y_READY + g));
                    if (leader) {
                        if (!wait_bar(ctl, bar(B_Y_READY + g), hcnt & 1)) ok = false;
                        tc_fence_after();
                        tma_store_3d(&tm_y, grp_w(g), h * kP, t0, bi);
                        bulk_commit();
                    }
                }
                ++hcnt;
            }
            if (!ok) break;
            flat += k;
        }
        if (leader) {
            bulk_wait0();
            // Tell the publisher there is nothing more to publish.  The leader alone signals it,
            // with all four arrivals at once, after its own last publication has been taken: an
            // arrival by another warp could otherwise complete the phase of that last publication
            // before the leader's arrival for it.
            if (npub >= 1) wait_bar(ctl, bar(B_PUB_DONE + g), (npub - 1) & 1);
            pubS[2 * g] = -1;
            mbar_arrive_cnt(bar(B_PUB_FULL + g), 4);
        }
        if (__any_sync(0xffffffffu, bad != 0) && lane == 0) set_status(p.status, SSD_ERR_DEVICE);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// ---- host side ----------------------------------------------------------------
int heads_per_item(const Problem &p) {
    const int hpg = (int)(p.H / p.G);
    int k = 1;
    for (int c = 1; c <= kMaxK; ++c)
        if (hpg % c == 0) k = c;
    return k;
}

// one counter per (batch, head, ring slot, 32 state rows)
size_t flags_bytes(const Problem &p) {
    return align_up(sizeof(unsigned) * (size_t)(p.b * p.H * 2 * (p.N / 32)), 256);
}

// Per-device launch setup, done once per device: SM count and the kernel's
// dynamic shared memory limit.  Returns the SM count (0 on failure).
int device_setup() {
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
        if (cudaFuncSetAttribute(ssd_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                cudaSuccess ||
            cudaFuncSetAttribute(ssd_fused_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
                cudaSuccess)
            return 0;
        sms[dev] = n;
    }
    return sms[dev];
}

}  // namespace

bool fused_supports(const Problem &p) {
    if (p.a_mode != SSD_A_SCALAR || p.io_dtype != SSD_DTYPE_BF16) return false;
    if (p.P != kP || (p.N != 128 && p.N != 256)) return false;
    if (p.Q != 128 && p.Q != 256) return false;
    if (p.T > (int64_t)INT32_MAX / 2 || p.b * p.H * 2 > (int64_t)INT32_MAX) return false;
    // the kernel indexes items and flat head numbers (items x heads per item) in 32 bits
    const int64_t blocks = (p.T + kBlk - 1) / kBlk;
    return blocks * p.b * p.H < (int64_t)INT32_MAX;
}

size_t fused_workspace_bytes(const Problem &p) {
    return kStatusBytes + flags_bytes(p) + sizeof(float) * (size_t)(p.b * p.H * 2 * p.N * kP);
}

cudaError_t fused_launch(const Problem &p, void *ws, size_t ws_bytes, cudaStream_t s) {
    (void)ws_bytes;
    char *base = static_cast<char *>(ws);
    FusedParams fp;
    fp.dt = p.dt;
    fp.A = p.A;
    fp.D = p.D;
    fp.init = p.init;
    fp.final_state = p.final_state;
    fp.status = reinterpret_cast<int *>(base);
    fp.ticket = reinterpret_cast<unsigned *>(base + 64);
    fp.flags = reinterpret_cast<unsigned *>(base + kStatusBytes);
    fp.ring = reinterpret_cast<float *>(base + kStatusBytes + flags_bytes(p));
    fp.b = (int)p.b;
    fp.T = (int)p.T;
    fp.H = (int)p.H;
    fp.G = (int)p.G;
    fp.k = heads_per_item(p);
    fp.HG = (int)(p.H / fp.k);
    fp.nblk = (int)((p.T + kBlk - 1) / kBlk);
    fp.total_items = fp.nblk * fp.b * fp.HG;
    const int64_t spin = debug_spin_limit();
    fp.chain_spin = spin > 0 ? spin : kDefaultChainSpin;
    fp.withhold = debug_withhold_chunk();

    fp.dt_tma = (fp.k % 4 == 0 && p.H % 4 == 0) ? 1 : 0;
    CUtensorMap mx, mB, mC, my, mdt;
    std::memset(&mdt, 0, sizeof(mdt));
    if (fp.dt_tma && !make_dt_map(&mdt, p.dt, (uint64_t)p.H, (uint64_t)p.T, (uint64_t)p.b, (uint32_t)fp.k))
        return cudaErrorInvalidValue;
    if (!make_map(&mx, p.x, (uint64_t)(p.H * p.P), (uint64_t)p.T, (uint64_t)p.b) ||
        !make_map(&mB, p.B, (uint64_t)(p.G * p.N), (uint64_t)p.T, (uint64_t)p.b) ||
        !make_map(&mC, p.C, (uint64_t)(p.G * p.N), (uint64_t)p.T, (uint64_t)p.b) ||
        !make_map(&my, p.y, (uint64_t)(p.H * p.P), (uint64_t)p.T, (uint64_t)p.b))
        return cudaErrorInvalidValue;

    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes + flags_bytes(p), s);
    if (e != cudaSuccess) return e;
    const int sms = device_setup();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = fp.total_items < sms ? fp.total_items : sms;
    record_dominant_start(s);
    if (p.N == 128)
        ssd_fused_kernel<1><<<grid, kThreads, kSmemBytes, s>>>(mx, mB, mC, my, mdt, fp);
    else
        ssd_fused_kernel<2><<<grid, kThreads, kSmemBytes, s>>>(mx, mB, mC, my, mdt, fp);
    record_dominant_stop(s);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssd
