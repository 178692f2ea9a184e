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
// The block's Gram terms, gate terms, T~ (16x16 forward substitution) and P are formed on CUDA
// cores in fp32.
//
// One persistent CTA of 320 threads per SM walks the (b, h) units:
//   state warpgroup (warps 0-3): thread j owns TMEM lane j (column j of S): moves S between
//     its shared-memory staging and TMEM, forms the split operands, sends o and the new S.
//   prep warpgroup (warps 4-7): the block's Gram, gate, T'' and P.
//   MMA warp (warp 8) and TMA producer (warp 9): the next unit's S (64 KB, a bulk copy into
//     one of two staging buffers) streams in while the current unit computes.
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
constexpr uint32_t S_BYTES = 65536;             // S of one unit, fp32 [d_k][d_v]
constexpr uint32_t OFF_S = 0;                    // 2 staging buffers
constexpr uint32_t OFF_KQ = 2 * S_BYTES;         // [K; Q]: 2 column blocks x 32 rows x 128 B, 128B swizzle
constexpr uint32_t OFF_V = OFF_KQ + 8192;        // V: 2 column blocks x 16 rows x 128 B
constexpr uint32_t OFF_TP = OFF_V + 4096;        // T'' hi, lo: 16 rows x 128 B each (first 32 B used)
constexpr uint32_t OFF_PP = OFF_TP + 4096;       // P hi, lo
constexpr uint32_t OFF_G = OFF_PP + 4096;        // fp32 kk[16][17], qk[16][17], then T~ [16][17]
constexpr uint32_t G_LD = 17;
constexpr uint32_t OFF_ROW = OFF_G + 3 * 16 * G_LD * 4;  // fp32 invn[16], gn[16]
constexpr uint32_t OFF_BAR = OFF_ROW + 128;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;      // tmem base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(OFF_KQ % 1024 == 0 && OFF_V % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_PP % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
static_assert(SMEM_ALLOC <= 232448, "exceeds the per-CTA shared memory limit");

// TMEM columns
constexpr uint32_t TM_S = 0;     // S^T fp32 (128)
constexpr uint32_t TM_SA = 128;  // S^T bf16 hi (64) | lo (64)
constexpr uint32_t TM_X = 256;   // X^T fp32 (16); then (-X)^T hi (8) | lo (8); then u^T hi | lo
constexpr uint32_t TM_O = 272;   // O^T fp32 (16), adjacent to TM_X: [X | O1] is one N = 32 product
constexpr uint32_t TM_U = 288;   // u^T fp32 (16)
constexpr uint32_t TM_COLS = 512;

constexpr int THREADS = 320;
constexpr int BAR_PREP = 2;
constexpr uint64_t WAIT_NS = 2000000000ull;

struct DtParams {
    CUtensorMap map_q, map_k, map_v;  // [B, m, H, 128] bf16: box 64 x 1 x 16 x 1, 128B swizzle
    const float *beta;                // [B, m, H]
    float *S;                         // [B, H, 128, 128]
    void *o;                          // [B, m, H, 128]
    int *status;
    int B, m, H;
    int euler;
    unsigned long long wait_ns;
};

struct Bars {
    uint64_t s_full[2], s_empty[2];  // S staging buffer landed / read (128 arrivals)
    uint64_t kqv_full, kqv_empty;    // K, Q, V of a block landed / no longer read
    uint64_t prep_ready, tp_free;    // T'', P of a block written / no longer read
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
        const float r0 = x[2 * c] - __uint_as_float(b0 & 0xffff0000u);
        const float r1 = x[2 * c + 1] - __uint_as_float(b1 & 0xffff0000u);
        lo[c] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
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
            mbar_init(&bars->s_empty[i], 128);
        }
        mbar_init(&bars->kqv_full, 1);
        mbar_init(&bars->kqv_empty, 1);
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
        const int j = tid;
        bool ok = true;
        int gb = 0;  // blocks processed (all units)
        int it = 0;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
            const int b = u / p.H, h = u % p.H;
            const int sb = it & 1;
            const float *stg = reinterpret_cast<const float *>(sm + OFF_S + sb * S_BYTES);
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                const int t0 = blk * MB, mb = min(MB, p.m - t0);
                if (blk == 0) {  // S^T of the unit from its staging: fp32 into TM_S and split into TM_SA
                    ok = dt_wait_warp(&bars->s_full[sb], (it >> 1) & 1, abort_flag, wait_ns);
                    if (!ok) break;
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
                    mbar_arrive(&bars->s_empty[sb]);  // the staging buffer may take the next S
                } else {  // S^T after the previous block's update -> split
                    ok = dt_wait_warp(&bars->s_done, (gb - 1) & 1, abort_flag, wait_ns);
                    if (!ok) break;
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
                tc_fence_before();
                mbar_arrive(&bars->sa_ready);
                ok = dt_wait_warp(&bars->x_done, gb & 1, abort_flag, wait_ns);
                if (!ok) break;
                tc_fence_after();
                {  // (-X)^T -> bf16 hi | lo (tokens past the block end are zero)
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
                }
                tc_fence_before();
                mbar_arrive(&bars->r_ready);
                ok = dt_wait_warp(&bars->u_done, gb & 1, abort_flag, wait_ns);
                if (!ok) break;
                tc_fence_after();
                {  // u^T -> bf16 hi | lo
                    float x[16];
                    uint32_t hi[8], lo[8];
                    tmem_ld16(lane_base + TM_U, x);
                    tmem_ld_wait();
                    split_pairs<8>(x, hi, lo);
                    tmem_st8u(lane_base + TM_X, hi);
                    tmem_st8u(lane_base + TM_X + 8, lo);
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&bars->u_ready);
                ok = dt_wait_warp(&bars->o_done, gb & 1, abort_flag, wait_ns);
                if (!ok) break;
                tc_fence_after();
                {  // o of the block's tokens (column j)
                    float ov[16];
                    tmem_ld16(lane_base + TM_O, ov);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        if (t < mb) {
                            const size_t row = ((size_t)b * p.m + t0 + t) * p.H + h;
                            if (OUT_BF16)
                                static_cast<__nv_bfloat16 *>(p.o)[row * D + j] = __float2bfloat16_rn(ov[t]);
                            else
                                static_cast<float *>(p.o)[row * D + j] = ov[t];
                        }
                    }
                }
            }
            if (!ok) break;
            {  // the unit's new S (its last block's o_done covers the state update)
                float *Su = p.S + (size_t)u * D * D;
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    float sv[32];
                    tmem_ld32(lane_base + TM_S + g * 32, sv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) Su[(size_t)(g * 32 + i) * D + j] = sv[i];
                }
            }
            tc_fence_before();
        }
        if (!ok) *abort_flag = 1;
    } else if (warp < 8) {
        // =============================== prep warpgroup ===============================
        const int pi = tid - 128;
        float *kk = reinterpret_cast<float *>(sm + OFF_G), *qk = kk + 16 * G_LD, *Tt = qk + 16 * G_LD;
        float *invn = reinterpret_cast<float *>(sm + OFF_ROW), *gn = invn + 16;
        const uint8_t *kq = sm + OFF_KQ;
        bool ok = true;
        int gb = 0;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int b = u / p.H, h = u % p.H;
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                const int t0 = blk * MB, mb = min(MB, p.m - t0);
                if (gb > 0) ok = dt_wait_warp(&bars->tp_free, (gb - 1) & 1, abort_flag, wait_ns);
                ok = ok && dt_wait_warp(&bars->kqv_full, gb & 1, abort_flag, wait_ns);
                if (named_bar_any(BAR_PREP, 128, !ok || *abort_flag)) {
                    ok = false;
                    break;
                }
                {  // Gram terms k_t.k_s and q_t.k_s (t = pi >> 3, s = 2 (pi & 7) + {0, 1}), fp32
                    const int t = pi >> 3, s = 2 * (pi & 7);
                    float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
#pragma unroll 4
                    for (int d8 = 0; d8 < D; d8 += 8) {
                        // 8 consecutive bf16 of rows t (K), 16 + t (Q), s, s + 1 (K)
                        const uint4 kt = *reinterpret_cast<const uint4 *>(kq + swz_offset(t, d8, 4096));
                        const uint4 qt = *reinterpret_cast<const uint4 *>(kq + swz_offset(16 + t, d8, 4096));
                        const uint4 ks0 = *reinterpret_cast<const uint4 *>(kq + swz_offset(s, d8, 4096));
                        const uint4 ks1 = *reinterpret_cast<const uint4 *>(kq + swz_offset(s + 1, d8, 4096));
                        const __nv_bfloat162 *pkt = reinterpret_cast<const __nv_bfloat162 *>(&kt);
                        const __nv_bfloat162 *pqt = reinterpret_cast<const __nv_bfloat162 *>(&qt);
                        const __nv_bfloat162 *pk0 = reinterpret_cast<const __nv_bfloat162 *>(&ks0);
                        const __nv_bfloat162 *pk1 = reinterpret_cast<const __nv_bfloat162 *>(&ks1);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 ft = __bfloat1622float2(pkt[e]), fq = __bfloat1622float2(pqt[e]);
                            const float2 f0 = __bfloat1622float2(pk0[e]), f1 = __bfloat1622float2(pk1[e]);
                            a0 = fmaf(ft.x, f0.x, fmaf(ft.y, f0.y, a0));
                            a1 = fmaf(ft.x, f1.x, fmaf(ft.y, f1.y, a1));
                            c0 = fmaf(fq.x, f0.x, fmaf(fq.y, f0.y, c0));
                            c1 = fmaf(fq.x, f1.x, fmaf(fq.y, f1.y, c1));
                        }
                    }
                    kk[t * G_LD + s] = a0;
                    kk[t * G_LD + s + 1] = a1;
                    qk[t * G_LD + s] = c0;
                    qk[t * G_LD + s + 1] = c1;
                }
                named_bar(BAR_PREP, 128);
                if (pi < 16) {  // gate terms of token t = pi (zero past the block end and for zero keys)
                    const int t = pi;
                    const float lam = kk[t * G_LD + t];
                    const float bt = t < mb ? p.beta[((size_t)b * p.m + t0 + t) * p.H + h] : 0.f;
                    const bool live = t < mb && lam > 0.f;
                    const float in = live ? rsqrtf(lam) : 0.f;
                    const float gam = !live ? 0.f : p.euler ? bt * lam : -expm1f(-bt * lam);
                    invn[t] = in;
                    gn[t] = gam * in;
                }
                named_bar(BAR_PREP, 128);
                if (pi < 16) {  // T~ = (I + A~)^{-1}, one lane per column c, the column in registers
                    const int c = pi;
                    float col[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) col[r] = r == c ? 1.f : 0.f;
#pragma unroll
                    for (int t = 1; t < 16; ++t) {
                        const float rt = gn[t];  // A~[t][s] = gamma_t/n_t * (k_t.k_s) / n_s
                        float acc = 0.f;
#pragma unroll
                        for (int s2 = 0; s2 < t; ++s2) acc = fmaf(rt * kk[t * G_LD + s2] * invn[s2], col[s2], acc);
                        col[t] = t > c ? -acc : col[t];
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) Tt[r * G_LD + c] = col[r];
                }
                named_bar(BAR_PREP, 128);
                {  // T'' = diag(1/n) T~ diag(gamma/n) and P = Q K^T o M, bf16 hi/lo, rows t, columns 8h8 .. 8h8+7
                    const int which = pi >> 5, t = (pi >> 1) & 15, h8 = pi & 1;  // which: 0 T'', 1 P; 64 threads idle
                    if (which < 2) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int s = 8 * h8 + e;
                            x[e] = which == 0 ? (s <= t ? invn[t] * Tt[t * G_LD + s] * gn[s] : 0.f)
                                              : (s <= t ? qk[t * G_LD + s] : 0.f);
                        }
                        uint32_t hh[4], ll[4];
                        split_pairs<4>(x, hh, ll);
                        uint8_t *dst = sm + (which == 0 ? OFF_TP : OFF_PP);
                        const uint32_t off = swz_offset(t, 8 * h8, 2048);
                        *reinterpret_cast<uint4 *>(dst + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        *reinterpret_cast<uint4 *>(dst + 2048 + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    }
                }
                fence_proxy_async_smem();
                named_bar(BAR_PREP, 128);
                if (pi == 0) mbar_arrive(&bars->prep_ready);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 8) {
        // =============================== MMA warp ===============================
        bool ok = true;
        int gb = 0;
        const uint32_t kq_s = s_sm + OFF_KQ, v_s = s_sm + OFF_V, tp = s_sm + OFF_TP, pp = s_sm + OFF_PP;
        const uint32_t id32 = idesc_bf16_f32(128, 32, 0, 0), id16 = idesc_bf16_f32(128, 16, 0, 0);
        const uint32_t id16v = idesc_bf16_f32(128, 16, 1, 0), id128k = idesc_bf16_f32(128, 128, 0, 1);
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                if (!(ok = dt_wait_warp(&bars->kqv_full, gb & 1, abort_flag, wait_ns))) break;
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
                mma_commit_e(&bars->kqv_empty);
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
    } else if (tid == 288) {
        // ============================ TMA producer (one thread) ============================
        prefetch_tensormap(&p.map_q);
        prefetch_tensormap(&p.map_k);
        prefetch_tensormap(&p.map_v);
        bool ok = true;
        int gb = 0, s_issued = 0, it = 0, kqv_issued = 0;
        auto load_s = [&](int unit_i, int idx) {  // S of unit unit_i into staging idx & 1
            const int sb = idx & 1;
            if (idx >= 2 && !(ok = dt_wait(&bars->s_empty[sb], ((idx - 2) >> 1) & 1, abort_flag, wait_ns))) return;
            mbar_arrive_expect_tx(&bars->s_full[sb], S_BYTES);
            const float *src = p.S + (size_t)unit_i * D * D;
            uint8_t *dst = sm + OFF_S + sb * S_BYTES;
            for (int q = 0; q < 4; ++q) bulk_load(dst + q * 16384, src + q * 4096, 16384, &bars->s_full[sb]);
            s_issued = idx + 1;
        };
        load_s(blockIdx.x, 0);
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
            const int b = u / p.H, h = u % p.H;
            if (u + (int)gridDim.x < units) load_s(u + gridDim.x, it + 1);  // the next unit's S streams in
            for (int blk = 0; blk < nblk && ok; ++blk, ++gb) {
                if (gb > 0 && !(ok = dt_wait(&bars->kqv_empty, (gb - 1) & 1, abort_flag, wait_ns))) break;
                mbar_arrive_expect_tx(&bars->kqv_full, 12288);
                const int t0 = blk * MB;
                for (int cb = 0; cb < 2; ++cb) {
                    tma_load_4d(sm + OFF_KQ + cb * 4096, &p.map_k, &bars->kqv_full, cb * 64, h, t0, b);
                    tma_load_4d(sm + OFF_KQ + cb * 4096 + 2048, &p.map_q, &bars->kqv_full, cb * 64, h, t0, b);
                    tma_load_4d(sm + OFF_V + cb * 2048, &p.map_v, &bars->kqv_full, cb * 64, h, t0, b);
                }
                kqv_issued = gb + 1;
            }
        }
        // every load in flight has landed before the CTA leaves (bounded; matters after an abort)
        for (int i = max(0, s_issued - 2); i < s_issued; ++i) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->s_full[i & 1], (i >> 1) & 1, 20000) && globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
        if (kqv_issued > 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->kqv_full, (kqv_issued - 1) & 1, 20000) &&
                   globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
        if (!ok) *abort_flag = 1;
    }

    if (*abort_flag && tid == 0) atomicExch(p.status, (int)EFLA_ERR_DEVICE_TIMEOUT);
    tc_fence_before();
    __syncthreads();
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

// [B, m, H, 128] bf16: box of 64 features x 1 head x 16 tokens x 1, 128-byte swizzle.
bool dt_map(CUtensorMap *mp, const void *ptr, int B, int m, int H) {
    auto fn = dt_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)m, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)m * H * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)MB, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
    if (!dt_map(&p.map_q, a.q, a.B, a.m, a.H) || !dt_map(&p.map_k, a.k, a.B, a.m, a.H) ||
        !dt_map(&p.map_v, a.v, a.B, a.m, a.H)) {
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
