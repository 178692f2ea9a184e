// Chunkwise EFLA forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The recurrence S_t = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T,
// o_t = S_t^T q_t ("Exact Flow Linear Attention" (gist.science), Metodologia 3;
// "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-4) is
// evaluated in chunks of C = 64 tokens with the WY/UT representation of the
// product of the chunk's rank-1 updates.  For one chunk with start state S
// (d_k x d_v, fp32), keys K, queries Q, values V (C x d), and per-row
//   lambda_t = ||k_t||^2,  n_t = sqrt(lambda_t),  gamma_t = 1 - e^{-beta_t lambda_t}
//   (gamma_t = alpha_t lambda_t; computed as -expm1(-beta_t lambda_t)):
//
//   A~  = strictly-lower( gamma_t (k_t . k_s) / (n_t n_s) )        (C x C)
//   T~  = (I + A~)^{-1}                                            (forward substitution)
//   T'  = T~ diag(gamma / n)
//   U^  = T' (V - K S)            u_t = U^_t / n_t   (= the rank-1 write u_t of token t)
//   O   = Q S + (Q K^T o M) u     (M lower-triangular INCLUDING the diagonal:
//                                  o_t reads the state after token t's update)
//   S  <- S + K^T u
//
// This follows from S_t = S_{t-1} + k_t u_t^T with u_t = alpha_t (v_t - S_{t-1}^T k_t):
// unrolling the chunk gives (I + A) U = diag(alpha)(V - K S) with
// A = strictly-lower(diag(alpha) K K^T) = D^{-1} A~ D, D = diag(n).  Working with
// unit-direction keys keeps every entry of A~ in [-1, 1] however much the key
// norms vary.
//
// Precision: the tensor-core operands that are not exact bf16 inputs (S, V - K S,
// T', u, Q K^T) are split into bf16 hi + lo parts and the products formed as
// hi*hi + hi*lo + lo*hi (or hi*x + lo*x against an exact bf16 input), with fp32
// accumulation in TMEM.  The state S lives in TMEM in fp32 for the whole
// sequence; T~ is computed in fp32 on the CUDA cores.
//
// Orientation: everything that involves the state is computed transposed, so
// that the state's d_v index is the MMA row (TMEM lane) and every operand is
// written by the thread that owns that lane:
//   [X^T | O1^T] = S^T [K ; Q]^T     (M = d_v = 128, N = 2C = 128, K = d_k = 128)
//   U^T          = (V - X)^T T'^T    (M = 128, N = C, K = C)
//   O^T         += u^T P^T,  P = Q K^T o M   (M = 128, N = C, K = C)
//   S^T         += u^T K             (M = 128, N = d_k = 128, K = C; K as MN-major operand)
// plus G = [K ; Q] K^T (M = 2C = 128, N = C, K = d_k) for the chunk-local Gram terms.
//
// One CTA of 128 threads (one warpgroup) per (sequence, head); thread j owns
// TMEM lane j.  K and Q tiles arrive by TMA (128B swizzle) double-buffered, the
// next chunk's load in flight while the current chunk is processed.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"

namespace efla {
namespace {
using namespace ptx;

constexpr int C = 64;
constexpr int D = 128;

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr uint32_t OFF_KQ = 0;             // 2 stages x [2 col blocks][128 rows][64] bf16; rows 0-63 K, 64-127 Q
constexpr uint32_t KQ_STAGE = 32768;
constexpr uint32_t OFF_ST_HI = 65536;      // S^T hi  [2][128 j][64 i]
constexpr uint32_t OFF_ST_LO = 98304;      // S^T lo
constexpr uint32_t OFF_RU_HI = 131072;     // (V - X)^T, then u^T, hi  [128 j][64 t]
constexpr uint32_t OFF_RU_LO = 147456;
constexpr uint32_t OFF_TP_HI = 163840;     // T' hi [64 t][64 s]
constexpr uint32_t OFF_TP_LO = 172032;
constexpr uint32_t OFF_P_HI = 180224;      // P hi [64 t][64 s]
constexpr uint32_t OFF_P_LO = 188416;
constexpr uint32_t OFF_AT = 196608;        // fp32 A~ rows split by column parity: [2][64 t][32]
constexpr uint32_t OFF_ROW = 212992;       // fp32 beta[64], gamma[64], inv_n[64], gn[64]
constexpr uint32_t OFF_BAR = 214016;       // mbarriers: tma[2], mma
constexpr uint32_t OFF_MISC = 214048;      // tmem base (u32), abort flag (i32)
constexpr uint32_t SMEM_ALLOC = 214064 + 1024;

// TMEM columns (fp32, lane = row of the MMA result)
constexpr uint32_t TM_S = 0;    // S^T            128 columns
constexpr uint32_t TM_X = 128;  // X^T = (K S)^T   64 columns
constexpr uint32_t TM_O = 192;  // O^T             64 columns
constexpr uint32_t TM_U = 256;  // U^^T            64 columns
constexpr uint32_t TM_G = 320;  // [K;Q] K^T       64 columns
constexpr uint32_t TM_COLS = 512;

constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s bound on any wait

struct TcParams {
    CUtensorMap map_q;
    CUtensorMap map_k;
    const __nv_bfloat16 *v;
    const float *beta;
    const float *S0;
    const int32_t *cu_seqlens;
    void *o;
    float *S_T;
    int *status;
    int B, T, H, N;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// Splits x into bf16 hi + lo (x ~= hi + lo to ~2^-17 relative).
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}

// Writes 64 fp32 values of one row as bf16 hi/lo into two 128B-swizzled tiles
// (row `row`, columns col0..col0+63; blocks of 64 columns `block` bytes apart).
__device__ __forceinline__ void store_row_split(uint8_t *hi_tile, uint8_t *lo_tile, int row, int col0,
                                                uint32_t block, const float *x) {
#pragma unroll
    for (int c = 0; c < 64; c += 8) {
        float h[8], l[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_bf16(x[c + e], h[e], l[e]);
        const uint32_t off = swz_offset(row, col0 + c, block);
        *reinterpret_cast<uint4 *>(hi_tile + off) =
            make_uint4(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]), pack_bf16(h[4], h[5]), pack_bf16(h[6], h[7]));
        *reinterpret_cast<uint4 *>(lo_tile + off) =
            make_uint4(pack_bf16(l[0], l[1]), pack_bf16(l[2], l[3]), pack_bf16(l[4], l[5]), pack_bf16(l[6], l[7]));
    }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&r)[64]) {
    float a[32], b[32];
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        r[i] = a[i];
        r[32 + i] = b[i];
    }
}

// All threads: CTA barrier with the tcgen05 ordering fences around it.
__device__ __forceinline__ void cta_sync_tc() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(128, 1) chunk_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *row_beta = reinterpret_cast<float *>(sm + OFF_ROW);
    float *row_gam = row_beta + 64;
    float *row_invn = row_beta + 128;
    float *row_gn = row_beta + 192;
    float *At = reinterpret_cast<float *>(sm + OFF_AT);
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_mma = bar_tma + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x / p.H, h = blockIdx.x % p.H;
    long b, bos, eos;
    if (p.cu_seqlens) {
        b = 0;
        bos = p.cu_seqlens[n];
        eos = p.cu_seqlens[n + 1];
        if (bos < 0 || eos < bos || eos > p.T) {  // malformed bounds: flag and touch nothing
            if (threadIdx.x == 0) atomicExch(p.status, (int)EFLA_ERR_INVALID_ARG);
            return;
        }
    } else {
        b = n;
        bos = 0;
        eos = p.T;
    }
    const int nchunks = eos > bos ? (int)((eos - bos + C - 1) / C) : 0;
    const size_t sbase = ((size_t)n * p.H + h) * D * D;
    const int j = tid;  // d_v index owned by this thread (TMEM lane)

    if (nchunks == 0) {  // empty sequence: S_T = S0
        if (p.S_T)
            for (int i = 0; i < D; ++i) p.S_T[sbase + (size_t)i * D + j] = p.S0 ? p.S0[sbase + (size_t)i * D + j] : 0.f;
        return;
    }

    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    cta_sync_tc();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t s_sm = smem_u32(sm);

    auto issue_tma = [&](int c) {
        const int stage = c & 1;
        uint8_t *dst = sm + OFF_KQ + stage * KQ_STAGE;
        const int tok = (int)(bos + (long)c * C);
        mbar_arrive_expect_tx(&bar_tma[stage], KQ_STAGE);
        for (int cb = 0; cb < 2; ++cb) {
            tma_load_4d(dst + cb * 16384, &p.map_k, &bar_tma[stage], cb * 64, h, tok, (int)b);
            tma_load_4d(dst + cb * 16384 + 8192, &p.map_q, &bar_tma[stage], cb * 64, h, tok, (int)b);
        }
    };
    if (tid == 0) {
        prefetch_tensormap(&p.map_q);
        prefetch_tensormap(&p.map_k);
        issue_tma(0);
    }

    // Initial state -> TMEM (S^T: lane j holds column j of S).
    {
        float r[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                r[i] = p.S0 ? p.S0[sbase + (size_t)(g * 32 + i) * D + j] : 0.f;
            tmem_st32(lane_base + TM_S + g * 32, r);
        }
        tmem_st_wait();
    }

    uint32_t mma_phase = 0;
    bool ok = true;
    int aborted_at = 0;
    auto wait_mma = [&]() {
        if (!mbar_wait(bar_mma, mma_phase, WAIT_NS)) ok = false;
        mma_phase ^= 1;
        tc_fence_after();
    };

    for (int c = 0; c < nchunks; ++c) {
        const int stage = c & 1;
        const long tok0 = bos + (long)c * C;
        const int valid = (int)min((long)C, eos - tok0);
        uint8_t *KQ = sm + OFF_KQ + stage * KQ_STAGE;
        const uint32_t kq_s = s_sm + OFF_KQ + stage * KQ_STAGE;

        // (a) values of this chunk for column j (kept as packed bf16 pairs), and the step sizes
        uint32_t vpk[C / 2];
        {
            const unsigned short *vv = reinterpret_cast<const unsigned short *>(p.v);
#pragma unroll
            for (int t = 0; t < C; t += 2) {
                const size_t row = ((size_t)b * p.T + (size_t)(tok0 + t)) * p.H + h;
                const uint32_t lo = t < valid ? vv[row * D + j] : 0u;
                const uint32_t hi = t + 1 < valid ? vv[(row + p.H) * D + j] : 0u;
                vpk[t / 2] = lo | (hi << 16);
            }
        }
        if (tid < C) {
            const size_t row = ((size_t)b * p.T + (size_t)(tok0 + tid)) * p.H + h;
            row_beta[tid] = tid < valid ? p.beta[row] : 0.f;
        }

        // (b) K and Q tiles
        if (!mbar_wait(&bar_tma[stage], (c >> 1) & 1, WAIT_NS)) ok = false;
        // (c) rows past the end of the sequence are zeroed (they may hold the next sequence)
        if (valid < C) {
            const int rows = C - valid;
            for (int e = tid; e < 4 * rows * 8; e += 128) {
                const int ch = e & 7, r = (e >> 3) % rows, part = (e >> 3) / rows;  // part: 0-1 K cb, 2-3 Q cb
                const int R = valid + r + ((part >> 1) ? 64 : 0), cb = part & 1;
                *reinterpret_cast<uint4 *>(KQ + cb * 16384 + (R >> 3) * 1024 + (R & 7) * 128 + ch * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
        }
        if (!ok) *abort_flag = 1;
        cta_sync_tc();
        if (*abort_flag) {
            aborted_at = c - 1;
            break;
        }

        // (d) next chunk's TMA; Gram MMA G = [K;Q] K^T
        if (tid == 0) {
            if (c + 1 < nchunks) issue_tma(c + 1);
            const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_bf16(tmem + TM_G, smem_desc(kq_s + off, 16, 1024), smem_desc(kq_s + off, 16, 1024), idesc,
                         ks > 0);
            }
            mma_commit(bar_mma);
        }
        wait_mma();

        // (e) per-row gate terms, A~ and P
        {
            float g[64];
            tmem_ld64(lane_base + TM_G, g);
            if (tid < C) {  // raw K K^T row t, parity-split
#pragma unroll
                for (int s = 0; s < 64; ++s) At[(s & 1) * 2048 + tid * 32 + (s >> 1)] = g[s];
            }
            __syncthreads();
            if (tid < C) {
                const int t = tid;
                const float lam = At[(t & 1) * 2048 + t * 32 + (t >> 1)];
                const float nrm = sqrtf(lam);
                const float invn = lam > 0.f ? 1.f / nrm : 0.f;
                const float gam = lam > 0.f ? -expm1f(-row_beta[t] * lam) : 0.f;
                row_gam[t] = gam;
                row_invn[t] = invn;
                row_gn[t] = gam * invn;
            }
            __syncthreads();
            if (tid < C) {
                const int t = tid;
                const float rs = row_gam[t] * row_invn[t];
#pragma unroll
                for (int s = 0; s < 64; ++s) {
                    float* a = &At[(s & 1) * 2048 + t * 32 + (s >> 1)];
                    *a = s < t ? rs * row_invn[s] * *a : 0.f;
                }
            } else {
                const int t = tid - C;
#pragma unroll
                for (int s = 0; s < 64; ++s) g[s] = s <= t ? g[s] : 0.f;
                store_row_split(sm + OFF_P_HI, sm + OFF_P_LO, t, 0, 8192, g);
            }
        }
        __syncthreads();

        // (f) T~ = (I + A~)^{-1}: thread (column cc, parity pp) holds T~[2m+pp][cc]
        {
            const int cc = (lane & 15) + 16 * warp;
            const int pp = lane >> 4;
            const float *Ap = At + pp * 2048;
            float col[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) col[m] = (2 * m + pp == cc) ? 1.f : 0.f;
#pragma unroll
            for (int t = 1; t < C; ++t) {
                const int mt = (t + 1) / 2;
                float acc = 0.f;
                const float *row = Ap + t * 32;
#pragma unroll
                for (int m = 0; m < mt; ++m) acc = fmaf(row[m], col[m], acc);
                const float tot = acc + __shfl_xor_sync(0xffffffffu, acc, 16);
                if ((t & 1) == pp && t > cc) col[t >> 1] = -tot;
            }
            // T' = T~ diag(gamma/n): scale column cc, write bf16 hi/lo into the B operand [t][s]
            const float gs = row_gn[cc];
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                float hi, lo;
                split_bf16(col[m] * gs, hi, lo);
                const uint32_t off = swz_offset(2 * m + pp, cc, 8192);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_TP_HI + off) = __float2bfloat16_rn(hi);
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_TP_LO + off) = __float2bfloat16_rn(lo);
            }
        }

        // (g) S^T -> bf16 hi/lo operand
        {
            float s64[64];
            tmem_ld64(lane_base + TM_S, s64);
            store_row_split(sm + OFF_ST_HI, sm + OFF_ST_LO, j, 0, 16384, s64);
            tmem_ld64(lane_base + TM_S + 64, s64);
            store_row_split(sm + OFF_ST_HI, sm + OFF_ST_LO, j, 64, 16384, s64);
        }
        fence_proxy_async_smem();
        cta_sync_tc();

        // (h) [X^T | O1^T] = S^T [K;Q]^T
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint32_t a_s = s_sm + (part ? OFF_ST_LO : OFF_ST_HI);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + TM_X, smem_desc(a_s + off, 16, 1024), smem_desc(kq_s + off, 16, 1024), idesc,
                             (part | ks) != 0);
                }
            }
            mma_commit(bar_mma);
        }
        wait_mma();

        // (i) R^T = V^T - X^T  -> operand; U^^T = R^T T'^T
        {
            float x[64];
            tmem_ld64(lane_base + TM_X, x);
#pragma unroll
            for (int t = 0; t < C; t += 2) {
                x[t] = __uint_as_float(vpk[t / 2] << 16) - x[t];
                x[t + 1] = __uint_as_float(vpk[t / 2] & 0xffff0000u) - x[t + 1];
            }
            store_row_split(sm + OFF_RU_HI, sm + OFF_RU_LO, j, 0, 16384, x);
        }
        fence_proxy_async_smem();
        cta_sync_tc();
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
            const uint32_t A_[3] = {OFF_RU_HI, OFF_RU_HI, OFF_RU_LO};
            const uint32_t B_[3] = {OFF_TP_HI, OFF_TP_LO, OFF_TP_HI};
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + TM_U, smem_desc(s_sm + A_[part] + ks * 32, 16, 1024),
                             smem_desc(s_sm + B_[part] + ks * 32, 16, 1024), idesc, (part | ks) != 0);
            mma_commit(bar_mma);
        }
        wait_mma();

        // (j) u^T = U^^T diag(1/n) -> operand; O^T += u^T P^T; S^T += u^T K
        {
            float u[64];
            tmem_ld64(lane_base + TM_U, u);
#pragma unroll
            for (int t = 0; t < C; ++t) u[t] *= row_invn[t];
            store_row_split(sm + OFF_RU_HI, sm + OFF_RU_LO, j, 0, 16384, u);
        }
        fence_proxy_async_smem();
        cta_sync_tc();
        if (tid == 0) {
            const uint32_t idesc_o = idesc_bf16_f32(128, 64, 0, 0);
            const uint32_t A_[3] = {OFF_RU_HI, OFF_RU_HI, OFF_RU_LO};
            const uint32_t B_[3] = {OFF_P_HI, OFF_P_LO, OFF_P_HI};
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + TM_O, smem_desc(s_sm + A_[part] + ks * 32, 16, 1024),
                             smem_desc(s_sm + B_[part] + ks * 32, 16, 1024), idesc_o, 1);
            const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + TM_S, smem_desc(s_sm + (part ? OFF_RU_LO : OFF_RU_HI) + ks * 32, 16, 1024),
                             smem_desc(kq_s + ks * 2048, 16384, 1024), idesc_s, 1);
            mma_commit(bar_mma);
        }
        wait_mma();

        // (k) outputs of this chunk
        {
            float ov[64];
            tmem_ld64(lane_base + TM_O, ov);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                if (t < valid) {
                    const size_t row = ((size_t)b * p.T + (size_t)(tok0 + t)) * p.H + h;
                    if (OUT_BF16)
                        static_cast<__nv_bfloat16 *>(p.o)[row * D + j] = __float2bfloat16_rn(ov[t]);
                    else
                        static_cast<float *>(p.o)[row * D + j] = ov[t];
                }
            }
        }
        if (!ok) *abort_flag = 1;
        cta_sync_tc();
        if (*abort_flag) {
            aborted_at = c;
            break;
        }
    }

    if (*abort_flag) {
        if (tid == 0) atomicExch(p.status, (int)EFLA_ERR_DEVICE_TIMEOUT);
        // let the most recently issued TMA land before the CTA exits (bounded)
        const int last = min(aborted_at + 1, nchunks - 1);
        mbar_wait(&bar_tma[last & 1], (last >> 1) & 1, WAIT_NS / 4);
    } else if (p.S_T) {
        float s64[64];
        tmem_ld64(lane_base + TM_S, s64);
#pragma unroll
        for (int i = 0; i < 64; ++i) p.S_T[sbase + (size_t)i * D + j] = s64[i];
        tmem_ld64(lane_base + TM_S + 64, s64);
#pragma unroll
        for (int i = 0; i < 64; ++i) p.S_T[sbase + (size_t)(64 + i) * D + j] = s64[i];
    }
    cta_sync_tc();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 4-D map over a [B, T, H, 128] bf16 tensor: box of 64 features x 1 head x 64 tokens.
bool make_map(CUtensorMap *m, const void *ptr, int B, int T, int H) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)C, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool OUT_BF16>
cudaError_t launch_typed(const TcParams &p, unsigned grid, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(chunk_tc_kernel<OUT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    chunk_tc_kernel<OUT_BF16><<<grid, 128, SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_tc(const FwdArgs &a, const char **why) {
    if (a.N == 0) return cudaSuccess;
    TcParams p;
    memset(&p, 0, sizeof p);
    if ((long long)a.B * a.T > 0) {
        if (!make_map(&p.map_q, a.q, a.B, a.T, a.H) || !make_map(&p.map_k, a.k, a.B, a.T, a.H)) {
            *why = "cuTensorMapEncodeTiled failed for q/k";
            return cudaErrorInvalidValue;
        }
    }
    p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.beta = a.beta;
    p.S0 = a.S0;
    p.cu_seqlens = a.cu_seqlens;
    p.o = a.o;
    p.S_T = a.S_T;
    p.status = device_status_ptr();
    p.B = a.B;
    p.T = a.T;
    p.H = a.H;
    p.N = a.N;
    if (!p.status) {
        *why = "device status word unavailable";
        return cudaErrorInvalidSymbol;
    }
    *why = "tcgen05 chunk kernel launch";
    const unsigned grid = (unsigned)((long)a.N * a.H);
    return a.o_dtype == EFLA_BF16 ? launch_typed<true>(p, grid, a.stream) : launch_typed<false>(p, grid, a.stream);
}

}  // namespace efla
