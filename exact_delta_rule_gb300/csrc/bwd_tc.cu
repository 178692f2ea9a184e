// State gradients of the chunked backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA):
// bf16 q, k with d_k = d_v = 128, chunks of 64, rows of [B, T].
//
// Reverse mode of the chunkwise forward ["Error-Free Linear Attention is a Free Lunch"
// (howistudyai), Step 4; "Exact Flow Linear Attention" (gist.science), Metodologia 3]: with
// dS' the gradient of the loss with respect to a chunk's end state, the chunk's start-state
// gradient is
//   G  = K dS' + P^T dO,      P = (Q K^T) o M_incl
//   dR = T''^T G,             T'' = diag(1/n) T~ diag(gamma/n) = (I + diag(alpha) L)^{-1} diag(alpha)
//   dS = dS' + Q^T dO - K^T dR
// and the chunks are walked from the last to the first, every dS' written out for the
// per-chunk gradient kernel.  The structure is the forward chunk kernel's, transposed the same
// way (dS^T fp32 in TMEM, lane j = column j, operands split into bf16 hi + lo):
//   G^T  = dS^T K^T + dO^T P         (N = 64; dO^T and P as MN-major operands)
//   dR^T = G^T T''                   (N = 64; T'' as an MN-major operand)
//   dS^T += dO^T Q - dR^T K          (N = 128; Q and K as MN-major operands)
// dO (fp32) enters as bf16 hi and lo arrays written by a pre-pass (split_do_kernel) and loaded
// by TMA like the other inputs.  G and dR (= dv) of every token are written out for the
// per-chunk gradient kernel, which then forms neither.
//
// One CTA of 320 threads per (b, h):
//   state warpgroup (warps 0-3): dS^T -> bf16 hi/lo operand (and dS' to HBM), G^T -> hi/lo (and
//     G to HBM), -dR^T -> hi/lo (and dv = dR, -dR as bf16 hi/lo to HBM);
//   prep warpgroup (warps 4-7): per chunk, the bf16 hi/lo tile of P from the Gram rows Q K^T in
//     TMEM (warps 6 and 7, TMEM lanes 64-127);
//   MMA warp (warp 8); TMA producer (warp 9): K, Q, dO hi/lo of chunk (reverse index) it into
//     stage it % 2, and the forward's T'' tile of that chunk (formed and written out by the
//     forward, run first with chunk-start states) into T''/P buffer it % 2.
// Every wait is bounded; on expiry the CTA records EFLA_ERR_DEVICE_TIMEOUT and leaves.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace efla {
namespace {
using namespace ptx;
using namespace tc;

constexpr int C = 64;
constexpr int D = 128;

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr int NSTAGE = 2;
constexpr uint32_t STAGE_BYTES = 65536;  // [K;Q] [2 cb][128 rows][64] (32 KB) + dO hi, lo [2 cb][64 rows][64] (16 KB each)
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_DOH = 32768;  // within a stage
constexpr uint32_t OFF_DOL = 49152;
// Per chunk parity: T'' hi, lo, then P hi, lo, each [64][64] bf16 (8 KB).
constexpr uint32_t OFF_TPP = NSTAGE * STAGE_BYTES;
constexpr uint32_t TPP_BYTES = 32768;
// -dR of a chunk as bf16 hi, then lo, [2 cb][64 rows][64] each (16 KB): the staging of its TMA stores
constexpr uint32_t OFF_DRS = OFF_TPP + 2 * TPP_BYTES;
constexpr uint32_t OFF_BAR = OFF_DRS + 32768;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;  // tmem base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(OFF_TPP % 1024 == 0 && OFF_DRS % 1024 == 0, "operand buffers must be 1024-byte aligned");
static_assert(SMEM_ALLOC <= 232448, "exceeds the per-CTA shared memory limit");

// TMEM columns
constexpr uint32_t TM_S = 0;     // dS^T fp32 (128)
constexpr uint32_t TM_SA = 128;  // dS^T bf16 hi (64) | lo (64); then dR^T fp32 (64)
constexpr uint32_t TM_X = 256;   // G^T fp32 (64); then G^T hi (32) | lo (32); then -dR^T hi | lo
constexpr uint32_t TM_G = 320;   // Gram rows [K; Q] K^T fp32 (64)
constexpr uint32_t TM_COLS = 512;

constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int BAR_PREP = 2;
constexpr int BAR_STATE = 3;

struct BtParams {
    CUtensorMap map_q, map_k, map_doh, map_dol;  // [B, T, H, 128] bf16: box 64 x 1 x 64 x 1, 128B swizzle
    CUtensorMap map_drh, map_drl;                // the same over -dR as bf16 hi and lo (stores)
    const float *beta;                           // [B, T, H]
    const float *dST;                            // [B, H, 128, 128] or nullptr (zero)
    float *dse;                                  // [B, H, nchunks] x 64 KB: dS' of every chunk as bf16 hi/lo
                                                 // operand tiles (put_col_split_tile)
    const uint8_t *tpp;                          // [B, H, nchunks] x 16 KB: the forward's T'' tiles
    float *dS0;                                  // [B, H, 128, 128] or nullptr
    float *g_out, *dr_out;                       // [B, T, H, 128] fp32: G and dR (= dv) of every token
    int *status;
    int B, T, H;
    int euler;
    int debug_stall;  // test hook: the MMA warp first waits on a barrier nothing completes
    unsigned long long wait_ns;
};

struct Bars {
    uint64_t tma_full[NSTAGE];  // K, Q, dO of a stage landed
    uint64_t s_free[NSTAGE];    // the stage's last reader (the state update) complete
    uint64_t g_done, g_free;    // Gram rows in TMEM / read by the prep
    uint64_t prep_ready[2];     // P of a chunk written and its T'' landed
    uint64_t t_full[2];         // the forward's T'' of a chunk landed (bulk copy)
    uint64_t tpp_free[2];       // the chunk's T''/P buffer no longer read
    uint64_t x_done, u_done, s_done;
    uint64_t sa_ready, r_ready, u_ready;  // state warpgroup operands written (128 arrivals)
    uint64_t drain[2];
    uint64_t never;             // never completed (the debug_stall test hook waits on it)
};
static_assert(sizeof(Bars) <= 256, "mbarrier block exceeds its slot");

// dO (fp32) -> bf16 hi (dO truncated) and lo (the remainder truncated), the split of the
// tensor-core operands; four elements per thread.
__global__ void __launch_bounds__(256) split_do_kernel(const float4 *__restrict__ dO, uint2 *__restrict__ hi,
                                                       uint2 *__restrict__ lo, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 x = __ldg(dO + i);
        uint32_t h[2], l[2];
        const float v[4] = {x.x, x.y, x.z, x.w};
        split_pack<2>(v, h, l);
        hi[i] = make_uint2(h[0], h[1]);
        lo[i] = make_uint2(l[0], l[1]);
    }
}

// A 64-column fp32 block of TMEM at lane_base + src (tokens 0-31 into x0, 32-63 into x1),
// times `sign`, as bf16 hi (columns 0-31) and lo (columns 32-63) at lane_base + TM_X.  Both
// halves are in registers before anything is written (src may be TM_X); x0 and x1 keep the
// values (before the sign) for the caller.
__device__ __forceinline__ void split64(uint32_t lane_base, uint32_t src, float sign, float (&x0)[32], float (&x1)[32]) {
    tmem_ld32(lane_base + src, x0);
    tmem_ld32(lane_base + src + 32, x1);
    tmem_ld_wait();
    uint32_t hi[16], lo[16];
    float y[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) y[t] = sign * x0[t];
    split_pack<16>(y, hi, lo);
    tmem_st16u(lane_base + TM_X, hi);
    tmem_st16u(lane_base + TM_X + 32, lo);
#pragma unroll
    for (int t = 0; t < 32; ++t) y[t] = sign * x1[t];
    split_pack<16>(y, hi, lo);
    tmem_st16u(lane_base + TM_X + 16, hi);
    tmem_st16u(lane_base + TM_X + 48, lo);
    tmem_st_wait();
}

// Column j of a chunk's [64 tokens][128] block of a [B, T, H, 128] fp32 tensor from registers
// (tokens past `valid` not written); consecutive threads write consecutive columns.
__device__ __forceinline__ void store_cols(float *base, size_t row_stride, int valid, const float (&x0)[32],
                                           const float (&x1)[32]) {
#pragma unroll
    for (int t = 0; t < 32; ++t)
        if (t < valid) base[(size_t)t * row_stride] = x0[t];
#pragma unroll
    for (int t = 0; t < 32; ++t)
        if (32 + t < valid) base[(size_t)(32 + t) * row_stride] = x1[t];
}

// Tokens 0-63 (x0: 0-31, x1: 32-63) of column j (this lane) of dR, negated, as bf16 hi and lo
// (split_pack's split) into the staging tiles at stg: [2 column blocks][64 tokens][64] bf16 with
// the 128-byte swizzle, hi then lo 16 KB on, the layout of the TMA boxes that store them.  Lanes
// j and j ^ 1 pair up: the even lane writes the hi word of columns j, j + 1, the odd lane the lo.
__device__ __forceinline__ void stage_neg_split(uint8_t *stg, int j, const float (&x0)[32], const float (&x1)[32]) {
    const bool odd = (j & 1) != 0;
    uint8_t *dst = stg + (odd ? 16384u : 0u);
#pragma unroll
    for (int t = 0; t < 64; ++t) {
        const float v = -(t < 32 ? x0[t] : x1[t - 32]);
        const uint32_t b = __float_as_uint(v);
        const uint32_t h16 = b >> 16;
        const uint32_t l16 = __float_as_uint(v - __uint_as_float(b & 0xffff0000u)) >> 16;
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? h16 : l16, 1);
        *reinterpret_cast<uint32_t *>(dst + swz_offset(t, j & ~1, 8192)) =
            odd ? (recv | (l16 << 16)) : (h16 | (recv << 16));
    }
}

__global__ void __launch_bounds__(320, 1) bwd_tc_kernel(const __grid_constant__ BtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint64_t wait_ns = p.wait_ns;
    const int b = blockIdx.x / p.H, h = blockIdx.x % p.H;
    const int nchunks = (p.T + C - 1) / C;  // >= 1 (the launcher skips T = 0)
    const size_t ubase = (size_t)blockIdx.x * D * D;
    // the it-th chunk processed is chunk nchunks - 1 - it (reverse order)
    auto chunk_of = [&](int it) { return nchunks - 1 - it; };

    if (tid == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&bars->tma_full[i], 1);
            mbar_init(&bars->s_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->prep_ready[i], 1);
            mbar_init(&bars->t_full[i], 1);
            mbar_init(&bars->tpp_free[i], 1);
            mbar_init(&bars->drain[i], 1);
        }
        mbar_init(&bars->g_done, 1);
        mbar_init(&bars->g_free, 1);
        mbar_init(&bars->x_done, 1);
        mbar_init(&bars->u_done, 1);
        mbar_init(&bars->s_done, 1);
        mbar_init(&bars->never, 1);
        mbar_init(&bars->sa_ready, 128);
        mbar_init(&bars->r_ready, 128);
        mbar_init(&bars->u_ready, 128);
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t s_sm = smem_u32(sm);

    if (tid >= 128 && tid < 256) {
        // =============================== prep warpgroup ===============================
        // Gram row r is TMEM lane r; rows 64-127 are Q K^T (P), read by warps 6 and 7.
        const int quarter = warp & 3;
        const int row = quarter * 32 + (tid & 31);
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool leader = tid == 128;
        // P of chunk (reverse index) it; hands the chunk over once its T'' (bulk-copied by the TMA
        // thread) has landed; false when the CTA aborts (the same answer in every prep thread)
        auto make_p = [&](int it, bool ok) -> bool {
            const int buf = it & 1;
            uint8_t *tpp_buf = sm + OFF_TPP + buf * TPP_BYTES;
            ok = ok && wait_bar_warp(&bars->g_done, it & 1, abort_flag, wait_ns);
            // this chunk's T''/P buffer was last read by the products of chunk it - 2
            if (it >= 2) ok = ok && wait_bar_warp(&bars->tpp_free[buf], ((it - 2) >> 1) & 1, abort_flag, wait_ns);
            tc_fence_after();
            // P[t][s] = Q K^T with the inclusive causal mask, bf16 hi/lo: rows 64-127 of the Gram
            // (rows 0-63, K K^T, are not needed), read into registers 32 columns at a time
            float g[2][32];
            if (ok && row >= C) {
                tmem_ld32(lane_base + TM_G, g[0]);
                tmem_ld32(lane_base + TM_G + 32, g[1]);
                tmem_ld_wait();
            }
            tc_fence_before();  // the next Gram may overwrite TM_G once every row is read
            if (named_bar_any(BAR_PREP, 128, !ok || *abort_flag)) {  // also spreads an abort
                *abort_flag = 1;
                return false;
            }
            if (leader) mbar_arrive(&bars->g_free);
            if (row >= C) {
                const int t = row - C;
                uint8_t *phi = tpp_buf + 16384, *plo = phi + 8192;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = 32 * hf + c8 + e <= t ? g[hf][c8 + e] : 0.f;
                        uint32_t hh[4], ll[4];
                        split_pack<4>(x, hh, ll);
                        const uint32_t off = swz_offset(t, 32 * hf + c8, 8192);
                        *reinterpret_cast<uint4 *>(phi + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        *reinterpret_cast<uint4 *>(plo + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    }
            }
            fence_proxy_async_smem();
            named_bar(BAR_PREP, 128);
            if (leader) {  // P written and T'' landed
                ok = wait_bar(&bars->t_full[buf], (it >> 1) & 1, abort_flag, wait_ns);
                mbar_arrive(&bars->prep_ready[buf]);
                if (!ok) *abort_flag = 1;
            }
            return true;
        };
        for (int it = 0; it < nchunks; ++it)
            if (!make_p(it, true)) break;
    } else if (tid < 128) {
        // =============================== state warpgroup ===============================
        const int j = tid;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        {  // dS_T -> TMEM (dS^T: lane j holds column j)
            float r[32];
#pragma unroll 1
            for (int g = 0; g < 4; g = opaque(g + 1)) {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = p.dST ? p.dST[ubase + (size_t)(g * 32 + i) * D + j] : 0.f;
                tmem_st32(lane_base + TM_S + g * 32, r);
            }
            tmem_st_wait();
        }
        bool ok = true;
        uint8_t *stg = sm + OFF_DRS;
        // A failed wait skips the work up to the chunk's consensus barrier, which every thread of
        // the warpgroup reaches, so that the warpgroup leaves together.
        for (int it = 0; it < nchunks; ++it) {
            if (it > 0) ok = wait_bar_warp(&bars->s_done, (it - 1) & 1, abort_flag, wait_ns);
            const int c = chunk_of(it), valid = min(C, p.T - c * C);
            const size_t row0 = ((size_t)b * p.T + (size_t)c * C) * p.H + h;
            float x0[32], x1[32];
            if (ok) {
                tc_fence_after();
                // dS^T -> bf16 hi/lo operand
#pragma unroll 1
                for (int g = 0; g < 4; g = opaque(g + 1)) {
                    float sv[32];
                    uint32_t hi[16], lo[16];
                    tmem_ld32(lane_base + TM_S + g * 32, sv);
                    tmem_ld_wait();
                    split_pack<16>(sv, hi, lo);
                    tmem_st16u(lane_base + TM_SA + g * 16, hi);
                    tmem_st16u(lane_base + TM_SA + 64 + g * 16, lo);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars->sa_ready);
                {  // dS' of this chunk (the gradient of its end state) to HBM while the tensor core
                   // forms G^T; TM_S changes again only after r_ready, which this warpgroup arrives at later
                    uint8_t *dst = reinterpret_cast<uint8_t *>(p.dse + ((size_t)blockIdx.x * nchunks + c) * D * D);
#pragma unroll 1
                    for (int g = 0; g < 4; g = opaque(g + 1)) {
                        float sv[32];
                        tmem_ld32(lane_base + TM_S + g * 32, sv);
                        tmem_ld_wait();
                        put_col_split_tile(dst, g * 32, j, sv);
                    }
                }
                ok = wait_bar_warp(&bars->x_done, it & 1, abort_flag, wait_ns);
            }
            if (ok) {
                tc_fence_after();
                split64(lane_base, TM_X, 1.f, x0, x1);  // G^T
                tc_fence_before();
                mbar_arrive(&bars->r_ready);
                // G for the per-chunk gradient kernel, sent while the tensor core forms dR
                store_cols(p.g_out + row0 * D + j, (size_t)p.H * D, valid, x0, x1);
                ok = wait_bar_warp(&bars->u_done, it & 1, abort_flag, wait_ns);
            }
            if (ok) {
                tc_fence_after();
                split64(lane_base, TM_SA, -1.f, x0, x1);  // -dR^T
                tc_fence_before();
                mbar_arrive(&bars->u_ready);
                store_cols(p.dr_out + row0 * D + j, (size_t)p.H * D, valid, x0, x1);  // dv = dR
            }
            // -dR as bf16 hi/lo for the per-chunk gradient kernel, staged in shared memory and
            // stored by TMA (rows past the sequence end are clipped) once the previous chunk's
            // stores have read the staging
            if (tid == 0) bulk_wait_read0();
            if (named_bar_any(BAR_STATE, 128, !ok)) {
                ok = false;
                break;
            }
            stage_neg_split(stg, j, x0, x1);
            fence_proxy_async_smem();
            named_bar(BAR_STATE, 128);
            if (tid == 0) {
                for (int cb = 0; cb < 2; ++cb) {
                    tma_store_4d(&p.map_drh, stg + cb * 8192, cb * 64, h, c * C, b);
                    tma_store_4d(&p.map_drl, stg + 16384 + cb * 8192, cb * 64, h, c * C, b);
                }
                bulk_commit();
            }
        }
        if (ok) {  // dS0: the gradient of the first chunk's start state
            ok = wait_bar_warp(&bars->s_done, (nchunks - 1) & 1, abort_flag, wait_ns);
            if (ok && p.dS0) {
                tc_fence_after();
#pragma unroll 1
                for (int g = 0; g < 4; g = opaque(g + 1)) {
                    float sv[32];
                    tmem_ld32(lane_base + TM_S + g * 32, sv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) p.dS0[ubase + (size_t)(g * 32 + i) * D + j] = sv[i];
                }
            }
        }
        if (tid == 0) bulk_wait0();  // the -dR stores have completed before the CTA leaves
        if (!ok) *abort_flag = 1;
    } else if (tid == 288) {
        // ============================ TMA producer (one thread) ============================
        prefetch_tensormap(&p.map_q);
        prefetch_tensormap(&p.map_k);
        prefetch_tensormap(&p.map_doh);
        prefetch_tensormap(&p.map_dol);
        int issued = 0, t_issued = 0;
        for (int it = 0; it < nchunks; ++it) {
            const int st = it % NSTAGE, buf = it & 1;
            // the forward's T'' of this chunk into its T''/P buffer, once chunk it - 2's products are
            // done with that buffer (the prep warpgroup waits for it before handing the chunk over)
            if (it >= 2 && !wait_bar(&bars->tpp_free[buf], ((it - 2) >> 1) & 1, abort_flag, wait_ns)) break;
            mbar_arrive_expect_tx(&bars->t_full[buf], 16384);
            bulk_load(sm + OFF_TPP + buf * TPP_BYTES, p.tpp + ((size_t)blockIdx.x * nchunks + chunk_of(it)) * 16384, 16384,
                      &bars->t_full[buf]);
            t_issued = it + 1;
            if (it >= NSTAGE && !wait_bar(&bars->s_free[st], ((it - NSTAGE) / NSTAGE) & 1, abort_flag, wait_ns)) break;
            uint8_t *dst = sm + OFF_STAGE + st * STAGE_BYTES;
            const int tok = chunk_of(it) * C;
            mbar_arrive_expect_tx(&bars->tma_full[st], STAGE_BYTES);
            for (int cb = 0; cb < 2; ++cb) {
                tma_load_4d(dst + cb * 16384, &p.map_k, &bars->tma_full[st], cb * 64, h, tok, b);
                tma_load_4d(dst + cb * 16384 + 8192, &p.map_q, &bars->tma_full[st], cb * 64, h, tok, b);
                tma_load_4d(dst + OFF_DOH + cb * 8192, &p.map_doh, &bars->tma_full[st], cb * 64, h, tok, b);
                tma_load_4d(dst + OFF_DOL + cb * 8192, &p.map_dol, &bars->tma_full[st], cb * 64, h, tok, b);
            }
            issued = it + 1;
        }
        // the last loads have landed before the CTA can leave (bounded; matters after an abort)
        for (int cc = max(0, issued - NSTAGE); cc < issued; ++cc) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->tma_full[cc % NSTAGE], (cc / NSTAGE) & 1, 20000) &&
                   globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
        for (int cc = max(0, t_issued - 2); cc < t_issued; ++cc) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->t_full[cc & 1], (cc >> 1) & 1, 20000) && globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
    } else if (warp == 8) {
        // =============================== MMA warp ===============================
        bool ok = true;
        int g_next = 0;
        // Gram rows [K; Q] K^T of chunks up to `limit`, each once the prep has read the previous
        // one and the chunk's stage has landed; with `block` false only what is ready now.
        auto issue_grams = [&](int limit, bool block) {
            while (ok && g_next <= limit && g_next < nchunks) {
                if (!block) {
                    const bool ready = (g_next == 0 || mbar_test(&bars->g_free, (g_next - 1) & 1)) &&
                                       mbar_test(&bars->tma_full[g_next % NSTAGE], (g_next / NSTAGE) & 1);
                    if (!__all_sync(0xffffffffu, ready)) break;
                } else {
                    if (g_next > 0 && !(ok = wait_bar_warp(&bars->g_free, (g_next - 1) & 1, abort_flag, wait_ns))) break;
                    if (!(ok = wait_bar_warp(&bars->tma_full[g_next % NSTAGE], (g_next / NSTAGE) & 1, abort_flag,
                                             wait_ns)))
                        break;
                }
                tc_fence_after();
                const uint32_t kq = s_sm + OFF_STAGE + (g_next % NSTAGE) * STAGE_BYTES;
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16_e(tmem + TM_G, smem_desc(kq + off, 16, 1024), smem_desc(kq + off, 16, 1024), idesc, ks > 0);
                }
                mma_commit_e(&bars->g_done);
                ++g_next;
            }
        };
        if (p.debug_stall) ok = wait_bar_warp(&bars->never, 0, abort_flag, wait_ns);
        issue_grams(0, true);
        for (int it = 0; it < nchunks && ok; ++it) {
            const int st = it % NSTAGE, buf = it & 1;
            const uint32_t kq_s = s_sm + OFF_STAGE + st * STAGE_BYTES;
            const uint32_t doh = kq_s + OFF_DOH, dol = kq_s + OFF_DOL;
            const uint32_t tp = s_sm + OFF_TPP + buf * TPP_BYTES, pb = tp + 16384;
            if (!(ok = wait_bar_warp(&bars->tma_full[st], (it / NSTAGE) & 1, abort_flag, wait_ns))) break;
            if (!(ok = wait_bar_warp(&bars->sa_ready, it & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            {  // G^T = dS^T K^T (the chain)
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16_ts_e(tmem + TM_X, tmem + TM_SA + part * 64 + ks * 8, smem_desc(kq_s + off, 16, 1024),
                                      idesc, (part | ks) != 0);
                    }
            }
            issue_grams(it + 1, false);
            if (!(ok = wait_bar_warp(&bars->prep_ready[buf], (it >> 1) & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            issue_grams(it + 1, true);
            if (!ok) break;
            {  // G^T += dO^T P: dO^T (M = j) and P (N = t) read as MN-major operands, K = s
                const uint32_t idesc = idesc_bf16_f32(128, 64, 1, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t ah = smem_desc(doh + ks * 2048, 8192, 1024), al = smem_desc(dol + ks * 2048, 8192, 1024);
                    const uint64_t bh = smem_desc(pb + ks * 2048, 8192, 1024), bl = smem_desc(pb + 8192 + ks * 2048, 8192, 1024);
                    mma_bf16_e(tmem + TM_X, ah, bh, idesc, 1);
                    mma_bf16_e(tmem + TM_X, ah, bl, idesc, 1);
                    mma_bf16_e(tmem + TM_X, al, bh, idesc, 1);
                }
                mma_commit_e(&bars->x_done);
            }
            if (!(ok = wait_bar_warp(&bars->r_ready, it & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            {  // dR^T = G^T T'' (T'' read as an MN-major operand, K = s), into TM_SA
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t th = smem_desc(tp + ks * 2048, 8192, 1024), tl = smem_desc(tp + 8192 + ks * 2048, 8192, 1024);
                    mma_bf16_ts_e(tmem + TM_SA, tmem + TM_X + ks * 8, th, idesc, ks > 0);
                    mma_bf16_ts_e(tmem + TM_SA, tmem + TM_X + ks * 8, tl, idesc, 1);
                    mma_bf16_ts_e(tmem + TM_SA, tmem + TM_X + 32 + ks * 8, th, idesc, 1);
                }
                mma_commit_e(&bars->u_done);
                mma_commit_e(&bars->tpp_free[buf]);
            }
            {  // dS^T += dO^T Q (after r_ready, so after the state warpgroup has sent this chunk's dS';
               // behind dR in the pipe, off the chain)
                const uint32_t idesc = idesc_bf16_f32(128, 128, 1, 1);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t bq = smem_desc(kq_s + 8192 + ks * 2048, 16384, 1024);
                    mma_bf16_e(tmem + TM_S, smem_desc(doh + ks * 2048, 8192, 1024), bq, idesc, 1);
                    mma_bf16_e(tmem + TM_S, smem_desc(dol + ks * 2048, 8192, 1024), bq, idesc, 1);
                }
            }
            issue_grams(it + 2, false);
            if (!(ok = wait_bar_warp(&bars->u_ready, it & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            {  // dS^T += (-dR)^T K (the chain; K read as an MN-major operand, K = t)
                const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_e(tmem + TM_S, tmem + TM_X + part * 32 + ks * 8,
                                      smem_desc(kq_s + ks * 2048, 16384, 1024), idesc, 1);
                mma_commit_e(&bars->s_done);
                mma_commit_e(&bars->s_free[st]);
            }
        }
        if (!ok) *abort_flag = 1;
        // every MMA this warp issued has completed before TMEM is released (bounded)
        mma_commit_e(&bars->drain[0]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait_sleep(&bars->drain[0], 0, 20000) && globaltimer_ns() - t0 < WAIT_NS) {
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();  // every role is done: an abort flagged by any of them is visible now
    if (*abort_flag && tid == 0) atomicExch(p.status, (int)EFLA_ERR_DEVICE_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 bt_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

}  // namespace

// [B, T, H, 128] bf16: box of 64 features x 1 head x 64 tokens x 1, 128-byte swizzle (the
// backward kernels' operand tiles).
bool bwd_row_map(CUtensorMap *m, const void *ptr, int B, int T, int H) {
    auto fn = bt_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)C, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// State gradients of the chunked backward on the tensor cores: bf16 q, k, d_k = d_v = 128,
// T > 0.  do_split: 2 x B*T*H*128 bf16 of scratch (dO hi, then lo); g_out: B*T*H*128 fp32
// (G of every token); dv receives dR.
cudaError_t launch_bwd_state_tc(const BwdArgs &a, float *dse, const uint8_t *tpp, void *do_split, float *g_out,
                                void *dr_split, const char **why) {
    const size_t n = (size_t)a.B * a.T * a.H * D;
    __nv_bfloat16 *hi = static_cast<__nv_bfloat16 *>(do_split), *lo = hi + n;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        *why = "querying the SM count";
        return e;
    }
    const size_t n4 = n / 4;
    const unsigned grid_split = (unsigned)std::min<size_t>((n4 + 255) / 256, (size_t)sms * 8);
    split_do_kernel<<<grid_split, 256, 0, a.stream>>>(reinterpret_cast<const float4 *>(a.dO),
                                                       reinterpret_cast<uint2 *>(hi), reinterpret_cast<uint2 *>(lo), n4);
    if ((e = cudaGetLastError()) != cudaSuccess) {
        *why = "dO split kernel launch";
        return e;
    }
    BtParams p;
    memset(&p, 0, sizeof p);
    if (!bwd_row_map(&p.map_q, a.q, a.B, a.T, a.H) || !bwd_row_map(&p.map_k, a.k, a.B, a.T, a.H) ||
        !bwd_row_map(&p.map_doh, hi, a.B, a.T, a.H) || !bwd_row_map(&p.map_dol, lo, a.B, a.T, a.H) ||
        !bwd_row_map(&p.map_drh, dr_split, a.B, a.T, a.H) ||
        !bwd_row_map(&p.map_drl, static_cast<__nv_bfloat16 *>(dr_split) + n, a.B, a.T, a.H)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    p.beta = a.beta;
    p.dST = a.dST;
    p.dse = dse;
    p.tpp = tpp;
    p.dS0 = a.dS0;
    p.g_out = g_out;
    p.dr_out = a.dv;
    p.status = device_status_ptr();
    p.B = a.B;
    p.T = a.T;
    p.H = a.H;
    p.euler = a.euler;
    p.wait_ns = wait_limit_ns();
    p.debug_stall = (debug_stall() & STALL_BWD_STATE) ? 1 : 0;
    static bool attr_done[64] = {};
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
        if (e != cudaSuccess) {
            *why = "setting the state-gradient kernel's shared memory";
            return e;
        }
        if (dev < 64) attr_done[dev] = true;
    }
    *why = "tcgen05 state-gradient kernel launch";
    bwd_tc_kernel<<<(unsigned)((long)a.B * a.H), 320, SMEM_ALLOC, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace efla
