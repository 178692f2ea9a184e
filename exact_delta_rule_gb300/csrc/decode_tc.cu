// Multi-token decode on the sm_103a tensor cores (tcgen05 + TMEM + TMA): m tokens per
// sequence appended to a resident state, S updated in place.
//
// Equal to m successive single-token steps of the recurrence
//   lambda = ||k||^2,  alpha = -expm1(-beta*lambda)/lambda (beta at lambda = 0),
//   S <- (I - alpha k k^T) S + alpha k v^T,  o = S^T q with the updated S
// ["Exact Flow Linear Attention" (gist.science), Metodologia 3; "Error-Free Linear
// Attention is a Free Lunch" (howistudyai), Steps 1-3 and "Putting it all together
// (pipeline)"].  The tokens of a sequence go in blocks of up to MB = 16, each block a chunk
// of the chunkwise form (howistudyai, Step 4):
//   u = T'' (V - K S),  T'' = diag(1/n) (I + A~)^{-1} diag(gamma/n),
//   A~ = strictly-lower( gamma_t (k_t . k_s) / (n_t n_s) )      (n_t = ||k_t||, gamma_t = alpha_t n_t^2)
//   O = Q S + (Q K^T o M) u          (M lower-triangular including the diagonal)
//   S <- S + K^T u
// so S is read from HBM once per call and written once.
//
// The products run on the tensor core in the transposed orientation of the chunk kernel
// (d_v is the MMA row and TMEM lane; S^T stays fp32 in TMEM), with the operands that are not
// exact bf16 inputs split into bf16 hi + lo parts (products hi*hi + hi*lo + lo*hi, or hi*x +
// lo*x against an exact input):
//   [X^T | O1^T] = S^T [K; Q]^T        (N = 32, K = d_k)
//   u^T = V^T T''^T + (-X)^T T''^T     (N = 16, K = 16; V^T read as an MN-major operand)
//   S^T += u^T K,  O^T = O1^T + u^T P^T,  P = Q K^T o M
// and the block's Gram terms [K; Q] K^T (N = 16, exact bf16 products summed in fp32; the MMA
// has M = 128 rows, of which the 32 rows of [K; Q] are kept).  The gate terms, T~ (16x16
// forward substitution) and the bf16 hi/lo packing of T'' and P are fp32 CUDA-core work.
//
// One persistent CTA of 256 threads per SM walks the (b, h) units:
//   state warpgroup (warps 0-3): thread j owns TMEM lane j (column j of S): moves S between its
//     shared-memory staging and TMEM, forms the split operands, writes o and the new S into
//     shared memory for the asynchronous stores.
//   prep warp (warp 4): the block's gate terms, T'' and P, from the Gram rows in TMEM.
//   MMA warp (warp 5).
//   K/Q/V producer (warp 6): the next block's K, Q, V (TMA, two stages) stream in while the
//     current block computes, so the Gram and prep of the next block run ahead of the state.
//   state mover (warp 7): per unit, a bulk copy of the new S (64 KB) from the staging buffer to
//     HBM, then the bulk load of the S two units ahead into the same buffer.
// Every wait is bounded; on expiry the CTA records EFLA_ERR_DEVICE_TIMEOUT and leaves.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"

namespace efla {
namespace {
using namespace ptx;

constexpr int D = 128;
constexpr int MB = 16;  // tokens per block

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr uint32_t S_BYTES = 65536;              // S of one unit, fp32 [d_k][d_v]
constexpr uint32_t OFF_S = 0;                     // 2 staging buffers
constexpr uint32_t KQ_BYTES = 8192;               // [K; Q]: 2 column blocks x 32 rows x 128 B, 128B swizzle
constexpr uint32_t V_BYTES = 4096;                // V: 2 column blocks x 16 rows x 128 B
constexpr uint32_t OFF_KQ = 2 * S_BYTES;          // 2 stages
constexpr uint32_t OFF_V = OFF_KQ + 2 * KQ_BYTES;  // 2 stages
constexpr uint32_t OFF_TP = OFF_V + 2 * V_BYTES;  // T'' hi, lo: 16 rows x 128 B each (first 32 B used)
constexpr uint32_t OFF_PP = OFF_TP + 4096;        // P hi, lo
constexpr uint32_t OFF_OT = OFF_PP + 4096;        // o tiles: 2 buffers x 8 KB (column blocks of 2 KB: 16 rows x 128 B)
constexpr uint32_t OFF_G = OFF_OT + 2 * 8192;     // fp32 A~ [16][17], T~ [16][17]
constexpr uint32_t G_LD = 17;
constexpr uint32_t OFF_ROW = OFF_G + 2 * 16 * G_LD * 4;  // fp32 invn[16], gn[16]
constexpr uint32_t OFF_BAR = OFF_ROW + 128;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;  // tmem base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(OFF_KQ % 1024 == 0 && OFF_V % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_PP % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
// The Gram MMA reads 128 rows of A from a [K; Q] stage, of which only the first 32 are kept:
// the rows past them must still lie inside the allocation.
static_assert(OFF_KQ + KQ_BYTES + 4096 + 16 * 1024 <= SMEM_USED, "Gram operand rows leave shared memory");
static_assert(SMEM_ALLOC <= 232448, "exceeds the per-CTA shared memory limit");

// TMEM columns
constexpr uint32_t TM_S = 0;     // S^T fp32 (128)
constexpr uint32_t TM_SA = 128;  // S^T bf16 hi (64) | lo (64)
constexpr uint32_t TM_X = 256;   // X^T fp32 (16); then (-X)^T hi (8) | lo (8); then u^T hi | lo
constexpr uint32_t TM_O = 272;   // O^T fp32 (16), adjacent to TM_X: [X | O1] is one N = 32 product
constexpr uint32_t TM_U = 288;   // u^T fp32 (16)
constexpr uint32_t TM_G = 304;   // Gram rows: lane t < 16 k_t . k_s, lane 16 + t q_t . k_s (16)
constexpr uint32_t TM_COLS = 512;

constexpr int THREADS = 256;
constexpr int TMA_TID = 192;
constexpr int SMOVE_TID = 224;
constexpr int BAR_STATE = 1;
constexpr uint64_t WAIT_NS = 2000000000ull;

struct DtParams {
    CUtensorMap map_q, map_k, map_v;  // [B, m, H, 128] bf16: box 64 x 1 x 16 x 1, 128B swizzle
    CUtensorMap map_o;                // [B, m, H, 128] in o's dtype: box (128 bytes) x 1 x 16 x 1, no swizzle
    const float *beta;                // [B, m, H]
    float *S;                         // [B, H, 128, 128]
    void *o;                          // [B, m, H, 128]
    int *status;
    int B, m, H;
    int euler;
    unsigned long long wait_ns;
};

struct Bars {
    uint64_t s_full[2], s_out[2];        // S staging buffer landed / holds the unit's new S (128 arrivals)
    uint64_t kqv_full[2], kqv_empty[2];  // K, Q, V stage landed / no longer read
    uint64_t g_done, g_free;             // Gram rows in TMEM / read by the prep warp
    uint64_t prep_ready, tp_free;        // T'', P of a block written / no longer read
    uint64_t sa_ready, x_done, r_ready, u_done, u_ready, s_done, o_done;
    uint64_t drain;
};
static_assert(sizeof(Bars) <= 256, "mbarrier block exceeds its slot");

__device__ __noinline__ bool dt_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint64_t limit) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort_flag = 1;
            return false;
        }
    }
}
__device__ __forceinline__ bool dt_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint64_t limit) {
    if (mbar_try_wait(bar, parity)) return true;
    return dt_wait_slow(bar, parity, abort_flag, limit);
}
__device__ __forceinline__ bool dt_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint64_t limit) {
    return __all_sync(0xffffffffu, dt_wait(bar, parity, abort_flag, limit));
}

// x = hi + lo as packed bf16 pairs (hi: x truncated to bf16; lo: the remainder truncated).
template <int NP>
__device__ __forceinline__ void split_pairs(const float *x, uint32_t *hi, uint32_t *lo) {
#pragma unroll
    for (int c = 0; c < NP; ++c) {
        const uint32_t b0 = __float_as_uint(x[2 * c]), b1 = __float_as_uint(x[2 * c + 1]);
        hi[c] = __byte_perm(b0, b1, 0x7632);
        // the two remainders x - hi (exact) in one packed fp32x2 fma: hi * (-1) + x
        const float2 r = __ffma2_rn(make_float2(__uint_as_float(b0 & 0xffff0000u), __uint_as_float(b1 & 0xffff0000u)),
                                    make_float2(-1.f, -1.f), make_float2(x[2 * c], x[2 * c + 1]));
        lo[c] = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
    }
}

// 16 fp32 values of row `row` of a 16-row operand tile (128B swizzle) as bf16 hi at `tile`, lo at tile + 2048.
__device__ __forceinline__ void put_row16(uint8_t *tile, int row, const float (&x)[16]) {
    uint32_t hh[8], ll[8];
    split_pairs<8>(x, hh, ll);
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
        const uint32_t off = swz_offset(row, 8 * h8, 2048);
        *reinterpret_cast<uint4 *>(tile + off) = make_uint4(hh[4 * h8], hh[4 * h8 + 1], hh[4 * h8 + 2], hh[4 * h8 + 3]);
        *reinterpret_cast<uint4 *>(tile + 2048 + off) =
            make_uint4(ll[4 * h8], ll[4 * h8 + 1], ll[4 * h8 + 2], ll[4 * h8 + 3]);
    }
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1) decode_tc_kernel(const __grid_constant__ DtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint64_t wait_ns = p.wait_ns;
    const int units = p.B * p.H;
    const int nblk = (p.m + MB - 1) / MB;
    if ((int)blockIdx.x >= units) return;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_out[i], 128);
            mbar_init(&bars->kqv_full[i], 1);
            mbar_init(&bars->kqv_empty[i], 1);
        }
        mbar_init(&bars->g_done, 1);
        mbar_init(&bars->g_free, 1);
        mbar_init(&bars->prep_ready, 1);
        mbar_init(&bars->tp_free, 1);
        mbar_init(&bars->sa_ready, 128);
        mbar_init(&bars->x_done, 1);
        mbar_init(&bars->r_ready, 128);
        mbar_init(&bars->u_done, 1);
        mbar_init(&bars->u_ready, 128);
        mbar_init(&bars->s_done, 1);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
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
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);

    if (warp < 4) {
        // =============================== state warpgroup ===============================
        // A failed wait skips the rest of the block's work but still reaches the block's
        // closing barrier, which every thread of the warpgroup passes before any leaves.
        const int j = tid;
        bool ok = true;
        int gb = 0;  // blocks processed (all units)
        int it = 0;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
            const int b = u / p.H, h = u % p.H;
            const int sb = it & 1;
            float *stg = reinterpret_cast<float *>(sm + OFF_S + sb * S_BYTES);
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                const int t0 = blk * MB, mb = min(MB, p.m - t0);
                if (blk == 0) {  // S^T of the unit from its staging: fp32 into TM_S and split into TM_SA
                    ok = dt_wait_warp(&bars->s_full[sb], (it >> 1) & 1, abort_flag, wait_ns);
                    if (ok) {
#pragma unroll 1
                        for (int g = 0; g < 4; ++g) {
                            float sv[32];
                            uint32_t hi[16], lo[16];
#pragma unroll
                            for (int i = 0; i < 32; ++i) sv[i] = stg[(g * 32 + i) * D + j];
                            tmem_st32(lane_base + TM_S + g * 32, sv);
                            split_pairs<16>(sv, hi, lo);
                            tmem_st16u(lane_base + TM_SA + g * 16, hi);
                            tmem_st16u(lane_base + TM_SA + 64 + g * 16, lo);
                        }
                        tmem_st_wait();
                    }
                } else {  // S^T after the previous block's update -> split
                    ok = dt_wait_warp(&bars->s_done, (gb - 1) & 1, abort_flag, wait_ns);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int g = 0; g < 4; ++g) {
                            float sv[32];
                            uint32_t hi[16], lo[16];
                            tmem_ld32(lane_base + TM_S + g * 32, sv);
                            tmem_ld_wait();
                            split_pairs<16>(sv, hi, lo);
                            tmem_st16u(lane_base + TM_SA + g * 16, hi);
                            tmem_st16u(lane_base + TM_SA + 64 + g * 16, lo);
                        }
                        tmem_st_wait();
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->sa_ready);
                ok = ok && dt_wait_warp(&bars->x_done, gb & 1, abort_flag, wait_ns);
                if (ok) {  // (-X)^T -> bf16 hi | lo (tokens past the block end are zero)
                    tc_fence_after();
                    float x[16];
                    uint32_t hi[8], lo[8];
                    tmem_ld16(lane_base + TM_X, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 16; ++t) x[t] = t < mb ? -x[t] : 0.f;
                    split_pairs<8>(x, hi, lo);
                    tmem_st8u(lane_base + TM_X, hi);
                    tmem_st8u(lane_base + TM_X + 8, lo);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bars->r_ready);
                }
                ok = ok && dt_wait_warp(&bars->u_done, gb & 1, abort_flag, wait_ns);
                if (ok) {  // u^T -> bf16 hi | lo
                    tc_fence_after();
                    float x[16];
                    uint32_t hi[8], lo[8];
                    tmem_ld16(lane_base + TM_U, x);
                    tmem_ld_wait();
                    split_pairs<8>(x, hi, lo);
                    tmem_st8u(lane_base + TM_X, hi);
                    tmem_st8u(lane_base + TM_X + 8, lo);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bars->u_ready);
                }
                ok = ok && dt_wait_warp(&bars->o_done, gb & 1, abort_flag, wait_ns);
                uint8_t *ot = sm + OFF_OT + (gb & 1) * 8192;
                if (ok) {  // o of the block's tokens (column j) into o tile gb & 1
                    tc_fence_after();
                    float ov[16];
                    tmem_ld16(lane_base + TM_O, ov);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        if (OUT_BF16)
                            *reinterpret_cast<__nv_bfloat16 *>(ot + (j >> 6) * 2048 + t * 128 + (j & 63) * 2) =
                                __float2bfloat16_rn(ov[t]);
                        else
                            *reinterpret_cast<float *>(ot + (j >> 5) * 2048 + t * 128 + (j & 31) * 4) = ov[t];
                    }
                    fence_proxy_async_smem();
                }
                if (named_bar_any(BAR_STATE, 128, !ok)) {
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                if (j == 0) {  // one thread stores the tile; rows past the sequence end fall outside the tensor
                    constexpr int NCB = OUT_BF16 ? 2 : 4, W = OUT_BF16 ? 64 : 32;
                    for (int cb = 0; cb < NCB; ++cb) tma_store_4d(&p.map_o, ot + cb * 2048, cb * W, h, t0, b);
                    bulk_commit();
                    // the tile is rewritten two blocks later, after the next closing barrier, which this
                    // thread reaches only once the copy has read it
                    bulk_wait_read0();
                }
            }
            if (!ok) break;
            {  // the unit's new S (its last block's o_done covers the state update) into its staging
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    float sv[32];
                    tmem_ld32(lane_base + TM_S + g * 32, sv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) stg[(g * 32 + i) * D + j] = sv[i];
                }
                fence_proxy_async_smem();
                mbar_arrive(&bars->s_out[sb]);
            }
            tc_fence_before();
        }
        if (j == 0) bulk_wait0();  // the o stores have completed
        if (!ok) *abort_flag = 1;
    } else if (warp == 4) {
        // ================================ prep warp ================================
        const int lane = tid & 31;
        float *At = reinterpret_cast<float *>(sm + OFF_G), *Tt = At + 16 * G_LD;
        float *invn = reinterpret_cast<float *>(sm + OFF_ROW), *gn = invn + 16;
        bool ok = true;
        int gb = 0;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int b = u / p.H, h = u % p.H;
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                const int t0 = blk * MB, mb = min(MB, p.m - t0);
                // beta of token `lane` (issued before the waits so that its latency overlaps them)
                const float bt = lane < mb ? p.beta[((size_t)b * p.m + t0 + lane) * p.H + h] : 0.f;
                if (!(ok = dt_wait_warp(&bars->g_done, gb & 1, abort_flag, wait_ns))) break;
                tc_fence_after();
                float row[16];  // lane t < 16: k_t . k_s; lane 16 + t: q_t . k_s
                tmem_ld16(tmem + TM_G, row);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->g_free);
                float lam = 0.f;
#pragma unroll
                for (int s = 0; s < 16; ++s) lam = s == lane ? row[s] : lam;
                {  // gate terms of token `lane` (zero past the block end and for zero keys)
                    const bool live = lane < mb && lam > 0.f;
                    const float in = live ? rsqrtf(lam) : 0.f;
                    const float gam = !live ? 0.f : p.euler ? bt * lam : -expm1f(-bt * lam);
                    if (lane < 16) {
                        invn[lane] = in;
                        gn[lane] = gam * in;
                    }
                }
                __syncwarp();
                if (lane < 16) {  // A~ row t = lane: gamma_t/n_t (k_t . k_s) / n_s, s < t
                    const float g_t = gn[lane];
#pragma unroll
                    for (int s = 0; s < 16; ++s) At[lane * G_LD + s] = s < lane ? g_t * row[s] * invn[s] : 0.f;
                }
                __syncwarp();
                if (lane < 16) {  // T~ = (I + A~)^{-1}, column c = lane, by forward substitution
                    const int c = lane;
                    float col[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) col[r] = r == c ? 1.f : 0.f;
#pragma unroll
                    for (int t = 1; t < 16; ++t) {
                        float acc = 0.f;
#pragma unroll
                        for (int s2 = 0; s2 < t; ++s2) acc = fmaf(At[t * G_LD + s2], col[s2], acc);
                        col[t] = t > c ? -acc : col[t];
                    }
                    const float gc = gn[c];
#pragma unroll
                    for (int r = 0; r < 16; ++r) Tt[r * G_LD + c] = col[r] * gc;
                }
                if (gb > 0 && !(ok = dt_wait_warp(&bars->tp_free, (gb - 1) & 1, abort_flag, wait_ns))) break;
                __syncwarp();
                {  // rows of T'' = diag(1/n) T~ diag(gamma/n) (lanes 0-15) and P = Q K^T o M (lanes 16-31)
                    const int t = lane & 15;
                    float x[16];
                    if (lane < 16) {
                        const float it = invn[t];
#pragma unroll
                        for (int s = 0; s < 16; ++s) x[s] = s <= t ? it * Tt[t * G_LD + s] : 0.f;
                    } else {
#pragma unroll
                        for (int s = 0; s < 16; ++s) x[s] = s <= t ? row[s] : 0.f;
                    }
                    put_row16(sm + (lane < 16 ? OFF_TP : OFF_PP), t, x);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->prep_ready);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 5) {
        // =============================== MMA warp ===============================
        bool ok = true;
        int gb = 0;
        const uint32_t tp = s_sm + OFF_TP, pp = s_sm + OFF_PP;
        const uint32_t id32 = idesc_bf16_f32(128, 32, 0, 0), id16 = idesc_bf16_f32(128, 16, 0, 0);
        const uint32_t id16v = idesc_bf16_f32(128, 16, 1, 0), id128k = idesc_bf16_f32(128, 128, 0, 1);
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                const int st = gb & 1;
                const uint32_t kq_s = s_sm + OFF_KQ + st * KQ_BYTES, v_s = s_sm + OFF_V + st * V_BYTES;
                if (!(ok = dt_wait_warp(&bars->kqv_full[st], (gb >> 1) & 1, abort_flag, wait_ns))) break;
                if (gb > 0 && !(ok = dt_wait_warp(&bars->g_free, (gb - 1) & 1, abort_flag, wait_ns))) break;
                tc_fence_after();
                // Gram rows [K; Q] K^T (rows 32-127 of the A operand are not used)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 4096 + (ks & 3) * 32;
                    mma_bf16_e(tmem + TM_G, smem_desc(kq_s + off, 16, 1024), smem_desc(kq_s + off, 16, 1024), id16,
                               ks > 0);
                }
                mma_commit_e(&bars->g_done);
                if (!(ok = dt_wait_warp(&bars->sa_ready, gb & 1, abort_flag, wait_ns))) break;
                tc_fence_after();
                // [X^T | O1^T] = S^T [K; Q]^T (N = 32 over the 32 rows of [K; Q])
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 4096 + (ks & 3) * 32;
                        mma_bf16_ts_e(tmem + TM_X, tmem + TM_SA + part * 64 + ks * 8, smem_desc(kq_s + off, 16, 1024),
                                      id32, (part | ks) != 0);
                    }
                mma_commit_e(&bars->x_done);
                if (!(ok = dt_wait_warp(&bars->prep_ready, gb & 1, abort_flag, wait_ns))) break;
                tc_fence_after();
                // u^T = V^T T''_hi^T + V^T T''_lo^T  (V^T as an MN-major operand: K = the 16 tokens)
                mma_bf16_e(tmem + TM_U, smem_desc(v_s, 2048, 1024), smem_desc(tp, 16, 1024), id16v, 0);
                mma_bf16_e(tmem + TM_U, smem_desc(v_s, 2048, 1024), smem_desc(tp + 2048, 16, 1024), id16v, 1);
                if (!(ok = dt_wait_warp(&bars->r_ready, gb & 1, abort_flag, wait_ns))) break;
                tc_fence_after();
                // u^T += (-X)_hi^T T''_hi^T + (-X)_hi^T T''_lo^T + (-X)_lo^T T''_hi^T
                mma_bf16_ts_e(tmem + TM_U, tmem + TM_X, smem_desc(tp, 16, 1024), id16, 1);
                mma_bf16_ts_e(tmem + TM_U, tmem + TM_X, smem_desc(tp + 2048, 16, 1024), id16, 1);
                mma_bf16_ts_e(tmem + TM_U, tmem + TM_X + 8, smem_desc(tp, 16, 1024), id16, 1);
                mma_commit_e(&bars->u_done);
                if (!(ok = dt_wait_warp(&bars->u_ready, gb & 1, abort_flag, wait_ns))) break;
                tc_fence_after();
                // S^T += u_hi^T K + u_lo^T K  (K as an MN-major operand: its 16 rows are the K dimension)
                mma_bf16_ts_e(tmem + TM_S, tmem + TM_X, smem_desc(kq_s, 4096, 1024), id128k, 1);
                mma_bf16_ts_e(tmem + TM_S, tmem + TM_X + 8, smem_desc(kq_s, 4096, 1024), id128k, 1);
                mma_commit_e(&bars->s_done);
                mma_commit_e(&bars->kqv_empty[st]);
                // O^T += u_hi^T P_hi^T + u_hi^T P_lo^T + u_lo^T P_hi^T
                mma_bf16_ts_e(tmem + TM_O, tmem + TM_X, smem_desc(pp, 16, 1024), id16, 1);
                mma_bf16_ts_e(tmem + TM_O, tmem + TM_X, smem_desc(pp + 2048, 16, 1024), id16, 1);
                mma_bf16_ts_e(tmem + TM_O, tmem + TM_X + 8, smem_desc(pp, 16, 1024), id16, 1);
                mma_commit_e(&bars->o_done);
                mma_commit_e(&bars->tp_free);
            }
        }
        if (!ok) *abort_flag = 1;
        mma_commit_e(&bars->drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait_sleep(&bars->drain, 0, 20000) && globaltimer_ns() - t0 < WAIT_NS) {
        }
        __syncwarp();
    } else if (tid == TMA_TID) {
        // ============================ TMA producer (one thread) ============================
        prefetch_tensormap(&p.map_q);
        prefetch_tensormap(&p.map_k);
        prefetch_tensormap(&p.map_v);
        bool ok = true;
        int gb = 0, kqv_issued = 0;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int b = u / p.H, h = u % p.H;
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                const int st = gb & 1;
                if (gb >= 2 && !(ok = dt_wait(&bars->kqv_empty[st], ((gb - 2) >> 1) & 1, abort_flag, wait_ns))) break;
                mbar_arrive_expect_tx(&bars->kqv_full[st], KQ_BYTES + V_BYTES);
                const int t0 = blk * MB;
                uint8_t *kq = sm + OFF_KQ + st * KQ_BYTES, *vv = sm + OFF_V + st * V_BYTES;
                for (int cb = 0; cb < 2; ++cb) {
                    tma_load_4d(kq + cb * 4096, &p.map_k, &bars->kqv_full[st], cb * 64, h, t0, b);
                    tma_load_4d(kq + cb * 4096 + 2048, &p.map_q, &bars->kqv_full[st], cb * 64, h, t0, b);
                    tma_load_4d(vv + cb * 2048, &p.map_v, &bars->kqv_full[st], cb * 64, h, t0, b);
                }
                kqv_issued = gb + 1;
            }
        }
        // every load in flight has landed before the CTA leaves (bounded; matters after an abort)
        for (int i = max(0, kqv_issued - 2); i < kqv_issued; ++i) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->kqv_full[i & 1], (i >> 1) & 1, 20000) &&
                   globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (tid == SMOVE_TID) {
        // ============================ state mover (one thread) ============================
        bool ok = true;
        int s_issued = 0;
        auto load_s = [&](int unit_i, int idx) {  // S of unit unit_i into staging idx & 1
            const int sb = idx & 1;
            mbar_arrive_expect_tx(&bars->s_full[sb], S_BYTES);
            const float *src = p.S + (size_t)unit_i * D * D;
            uint8_t *dst = sm + OFF_S + sb * S_BYTES;
            for (int q = 0; q < 4; ++q) bulk_load(dst + q * 16384, src + q * 4096, 16384, &bars->s_full[sb]);
            s_issued = idx + 1;
        };
        load_s(blockIdx.x, 0);
        if ((int)(blockIdx.x + gridDim.x) < units) load_s(blockIdx.x + gridDim.x, 1);
        int it = 0;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
            const int sb = it & 1;
            if (!(ok = dt_wait(&bars->s_out[sb], (it >> 1) & 1, abort_flag, wait_ns))) break;
            uint8_t *src = sm + OFF_S + sb * S_BYTES;
            float *dst = p.S + (size_t)u * D * D;
            for (int q = 0; q < 4; ++q) bulk_store(dst + q * 4096, src + q * 16384, 16384);
            bulk_commit();
            bulk_wait_read0();  // the buffer is free once the copy has read it
            const int u2 = u + 2 * (int)gridDim.x;
            if (u2 < units) load_s(u2, it + 2);
        }
        bulk_wait0();
        // every load in flight has landed before the CTA leaves (bounded; matters after an abort)
        for (int i = max(0, s_issued - 2); i < s_issued; ++i) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->s_full[i & 1], (i >> 1) & 1, 20000) && globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
        if (!ok) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();  // every role is done: an abort flagged by any of them is visible now
    if (*abort_flag && tid == 0) atomicExch(p.status, (int)EFLA_ERR_DEVICE_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 dt_encode_fn() {
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

// [B, m, H, 128] of 2-byte (bf16) or 4-byte (fp32) elements: a box of 128 bytes of features x
// 1 head x 16 tokens x 1; inputs with the 128-byte swizzle of the MMA operands, o unswizzled.
bool dt_map(CUtensorMap *mp, const void *ptr, int B, int m, int H, bool f32, bool swizzle) {
    auto fn = dt_encode_fn();
    if (!fn) return false;
    const cuuint64_t es_b = f32 ? 4 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)m, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * es_b, (cuuint64_t)H * D * es_b, (cuuint64_t)m * H * D * es_b};
    cuuint32_t box[4] = {(cuuint32_t)(128 / es_b), 1, (cuuint32_t)MB, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(mp, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool OUT_BF16>
cudaError_t dt_launch(const DtParams &p, unsigned grid, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_tc_kernel<OUT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_done[dev] = true;
    }
    decode_tc_kernel<OUT_BF16><<<grid, THREADS, SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

// Multi-token decode on the tensor cores: bf16 q, k, v with d_k = d_v = 128.
cudaError_t launch_decode_tokens_tc(const DecodeArgs &a, const char **why) {
    if (a.B == 0 || a.m == 0) return cudaSuccess;
    DtParams p;
    memset(&p, 0, sizeof p);
    if (!dt_map(&p.map_q, a.q, a.B, a.m, a.H, false, true) || !dt_map(&p.map_k, a.k, a.B, a.m, a.H, false, true) ||
        !dt_map(&p.map_v, a.v, a.B, a.m, a.H, false, true) ||
        !dt_map(&p.map_o, a.o, a.B, a.m, a.H, a.o_dtype != EFLA_BF16, false)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    p.beta = a.beta;
    p.S = a.S;
    p.o = a.o;
    p.status = device_status_ptr();
    p.B = a.B;
    p.m = a.m;
    p.H = a.H;
    p.euler = a.euler;
    p.wait_ns = wait_limit_ns();
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        *why = "querying the SM count";
        return e;
    }
    const long units = (long)a.B * a.H;
    const unsigned grid = (unsigned)std::min<long>(units, sms);
    *why = "tcgen05 decode kernel launch";
    return a.o_dtype == EFLA_BF16 ? dt_launch<true>(p, grid, a.stream) : dt_launch<false>(p, grid, a.stream);
}

}  // namespace efla
