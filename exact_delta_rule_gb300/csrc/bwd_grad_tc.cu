// Per-chunk gradients of the chunked backward on the sm_103a tensor cores (tcgen05 + TMEM):
// bf16 q, k, v with d_k = d_v = 128, chunks of 64, after the tensor-core state pass.
//
// Reverse mode of the chunkwise forward ["Error-Free Linear Attention is a Free Lunch"
// (howistudyai), Step 4; "Exact Flow Linear Attention" (gist.science), Metodologia 3].  For a
// chunk with start state S, end-state gradient dS', and G, dR (= dv) from the state pass, with
// L = strictly-lower(K K^T) and T'' = T diag(alpha) the forward's:
//   R  = V - K S,  U = T'' R
//   dY = G - L^T dR,  Z = R - L U,  dalpha_t = sum_j dY[t][j] Z[t][j]
//   dP = (dO U^T) o M_incl,  dL = -strictly-lower(dR U^T)
//   dq = dO S^T + dP K
//   dk = -dR S^T + U dS'^T + dP^T Q + (dL + dL^T + diag(2 dalpha dalpha/dlambda)) K
//   dbeta = dalpha (dalpha/dbeta)
// All products run on the tensor core in the transposed orientation (TMEM lane = feature),
// every operand that is not an exact bf16 input split into bf16 hi + lo (fp32 accumulation):
//   P0  Gram K K^T (TMEM); gate terms; -L as a bf16 hi/lo tile (T'' is the forward's, loaded whole;
//       a zero key's diagonal entry, 0 there, is set to alpha_t here)
//   P1  X^T = S^T K^T;  [dQ^T | dK^T] = S [dO; -dR]^T            (S: a swizzled bf16 tile)
//   P2  R^T = V^T - X^T (TMEM);  U^T = R^T T''^T
//   P3  Z^T = R^T + U^T (-L)^T;  -dY^T = -G^T + (-dR)^T (-L)        ((-dR)^T read from the tile)
//       [dP; -dR U^T] = [dO; -dR] U^T;  dK^T += dS' U^T          (dS': the same tile, reloaded)
//   P4  dalpha (lane reduction of -dY^T o Z^T); dP and E = dL + dL^T + diag(2 dalpha dalpha/dlambda)
//       as bf16 hi/lo tiles
//   P5  dQ^T += K^T dP^T;  dK^T += Q^T dP + K^T E
//   P6  dq, dk, dbeta to HBM
// Persistent CTAs of 288 threads walk the (b, h, chunk) items with a stride of the grid:
//   warps 0-7 (CUDA cores): every step above that is not a product, the two warpgroups each on
//     half of a chunk's 64 tokens; they meet at named barrier 1 only and hand operands to the
//     tensor core through mbarriers;
//   warp 8 (one lane): TMA loads of K, Q, dO and -dR (the last two as bf16 hi/lo arrays), bulk
//     copies of the S and dS' tiles (written in this layout by the forward and the state pass),
//     every tcgen05.mma and commit.
// Every wait is bounded; on expiry the CTA records EFLA_ERR_DEVICE_TIMEOUT and leaves.
#include <cudaTypedefs.h>

#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace efla {
namespace {
using namespace ptx;
using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NW = 256;         // CUDA-core threads (warps 0-7)
constexpr int NTH = NW + 32;    // and the MMA / TMA warp
constexpr int BAR_W = 1;        // named barrier of the CUDA-core warps

// Shared memory map (bytes from a 1024-byte aligned base).  Operand tiles are bf16 with the
// 128-byte swizzle in column blocks of 64 elements; "hi | lo" pairs are the two split parts.
constexpr uint32_t OFF_KQ = 0;        // [K; Q]: 2 column blocks x 128 rows (K 0-63, Q 64-127), 32 KB
constexpr uint32_t OFF_DOR = 32768;   // [dO; -dR] hi | lo: 2 column blocks x 128 rows each, 64 KB; later fp32 dL [64][65]
constexpr uint32_t OFF_SS = 98304;    // S, later dS', hi | lo: 2 column blocks x 128 rows each, 64 KB
constexpr uint32_t OFF_W = 163840;    // T'' hi | lo [64][64] (16 KB, the forward's); later dP hi | lo
constexpr uint32_t OFF_L = 180224;    // -L hi | lo [64][64] (16 KB); later E hi | lo
constexpr uint32_t OFF_UT = 196608;   // U^T hi | lo [128][64] (32 KB)
constexpr uint32_t OFF_ROW = 229376;  // fp32 per token: dalpha/dbeta, dalpha/dlambda, dalpha
constexpr uint32_t OFF_BAR = OFF_ROW + 3 * C * 4;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;  // tmem base, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
constexpr int DL_LD = 65;
constexpr uint32_t LO_128 = 32768;  // lo part after hi in the 128 x 128 tiles
constexpr uint32_t LO_UT = 16384;   // ... in the U^T tile
constexpr uint32_t LO_64 = 8192;    // ... in the 64 x 64 tiles
static_assert(OFF_DOR % 1024 == 0 && OFF_SS % 1024 == 0 && OFF_W % 1024 == 0 && OFF_L % 1024 == 0 &&
                  OFF_UT % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
static_assert(OFF_DOR == OFF_KQ + 32768 && OFF_SS == OFF_DOR + 2 * LO_128 && OFF_W == OFF_SS + 2 * LO_128 &&
                  OFF_L == OFF_W + 2 * LO_64 && OFF_UT == OFF_L + 2 * LO_64 && OFF_ROW == OFF_UT + 2 * LO_UT,
              "regions overlap");
static_assert(C * DL_LD * 4 <= 2 * LO_128, "fp32 scratch exceeds its region");
static_assert(SMEM_ALLOC <= 232448, "exceeds the per-CTA shared memory limit");

// TMEM columns (fp32 unless split: bf16 pairs, hi in the first 32 columns, lo in the next 32)
constexpr uint32_t TM_P = 0;     // [dP; -dR U^T] (64)
constexpr uint32_t TM_X = 128;   // X^T -> R^T -> Z^T (64)
constexpr uint32_t TM_RS = 192;  // R^T split (64)
constexpr uint32_t TM_U = 256;   // Gram -> U^T -> -G^T -> -dY^T (64)
constexpr uint32_t TM_US = 320;  // U^T split (64)
constexpr uint32_t TM_DQ = 384;  // dQ^T (64)
constexpr uint32_t TM_DK = 448;  // dK^T (64), adjacent to dQ^T: one N = 128 product fills both
constexpr uint32_t TM_COLS = 512;

constexpr uint64_t DRAIN_NS = 2000000000ull;

struct GtParams {
    CUtensorMap map_q, map_k, map_doh, map_dol, map_drh, map_drl;  // [B, T, H, 128] bf16: box 64 x 1 x 64 x 1,
                                                                   // 128B swizzle (dO, -dR as hi and lo)
    const __nv_bfloat16 *v;                      // [B, T, H, 128]
    const float *beta;                           // [B, T, H]
    const uint8_t *states, *dse;                 // [B, H, nchunks] x 64 KB: S and dS' of every chunk as
                                                 // bf16 hi/lo operand tiles (put_col_split_tile)
    const uint8_t *tpp;                          // [B, H, nchunks] x 16 KB: the forward's T'' tiles
    const float *g;                              // [B, T, H, 128]: G of every token
    float *dq, *dk, *dbeta;
    int *status;
    int T, H, items;                             // items = B H nchunks
    int euler;
    int debug_stall;  // test hook: the MMA warp first waits on a barrier nothing completes
    unsigned long long wait_ns;
};

struct Bars {
    uint64_t tma_kq, tma_dor;              // K, Q / dO, -dR of the item landed (TMA)
    uint64_t s_full, d_full, t_full;       // the S / dS' / T'' tile landed (bulk copies)
    uint64_t g, m1a, m1b, u, a, b, m2;     // products complete (tcgen05.commit)
    uint64_t w_u, w_p3, w_p5, w_free;      // operands written / TMEM read by the CUDA-core warps (8 arrivals)
    uint64_t drain;
    uint64_t never;                        // never completed (the debug_stall test hook waits on it)
};
static_assert(sizeof(Bars) <= 256, "mbarrier block exceeds its slot");

// x[0..15] as bf16 hi and lo of row `row`, columns col0 .. col0 + 15 (col0 + 15 < 64) of a
// swizzled tile (hi at `tile`, lo at tile + lo_off).
__device__ __forceinline__ void put16(uint8_t *tile, uint32_t lo_off, int row, int col0, const float *x) {
    uint32_t hh[8], ll[8];
    split_pack<8>(x, hh, ll);
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
        const uint32_t off = swz_offset(row, col0 + 8 * h8, 0);
        *reinterpret_cast<uint4 *>(tile + off) = make_uint4(hh[4 * h8], hh[4 * h8 + 1], hh[4 * h8 + 2], hh[4 * h8 + 3]);
        *reinterpret_cast<uint4 *>(tile + lo_off + off) =
            make_uint4(ll[4 * h8], ll[4 * h8 + 1], ll[4 * h8 + 2], ll[4 * h8 + 3]);
    }
}

// 32 fp32 values (this warpgroup's 32 tokens) as a TMEM A operand: bf16 pairs, hi at
// base + 16 h, lo at base + 32 + 16 h.
__device__ __forceinline__ void tsplit32(uint32_t lane_base, uint32_t base, int h, const float (&x)[32]) {
    uint32_t hh[16], ll[16];
    split_pack<16>(x, hh, ll);
    tmem_st16u(lane_base + base + 16 * h, hh);
    tmem_st16u(lane_base + base + 32 + 16 * h, ll);
}

// Sum over the 32 lanes of a warp of x[0..31]: lane l returns the sum of x[l] (reduce-scatter
// by halving, 31 shuffles).
__device__ __forceinline__ float lane_reduce_scatter(float (&x)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = up ? x[i] : x[i + w];
            const float keep = up ? x[i + w] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return x[0];
}


// One work item: chunk c of unit (b, h); token t of the chunk is row row0 + t H of [B, T, H].
struct Item {
    int b, h, t0, valid;
    size_t row0;
};
__device__ __forceinline__ Item item_of(const GtParams &p, int w, int nc) {
    Item it;
    const int unit = w / nc, c = w - unit * nc;
    it.b = unit / p.H;
    it.h = unit - it.b * p.H;
    it.t0 = c * C;
    it.valid = min(C, p.T - it.t0);
    it.row0 = ((size_t)it.b * p.T + (size_t)it.t0) * p.H + it.h;
    return it;
}

__global__ void __launch_bounds__(NTH, 1) bwd_grad_tc_kernel(const __grid_constant__ GtParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = (p.T + C - 1) / C;
    const uint64_t wait_ns = p.wait_ns;
    const uint32_t s_sm = smem_u32(sm);

    if (tid == 0) {
        mbar_init(&bars->tma_kq, 1);
        mbar_init(&bars->tma_dor, 1);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->d_full, 1);
        mbar_init(&bars->t_full, 1);
        mbar_init(&bars->g, 1);
        mbar_init(&bars->m1a, 1);
        mbar_init(&bars->m1b, 1);
        mbar_init(&bars->u, 1);
        mbar_init(&bars->a, 1);
        mbar_init(&bars->b, 1);
        mbar_init(&bars->m2, 1);
        mbar_init(&bars->w_u, 8);
        mbar_init(&bars->w_p3, 8);
        mbar_init(&bars->w_p5, 8);
        mbar_init(&bars->w_free, 8);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->never, 1);
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

    if (warp == 8) {
        // ============================ MMA / TMA warp ============================
        const bool leader = lane == 0;
        const uint32_t kq = s_sm + OFF_KQ, dor = s_sm + OFF_DOR, ss = s_sm + OFF_SS;
        const uint32_t wt = s_sm + OFF_W, l = s_sm + OFF_L, ut = s_sm + OFF_UT;
        if (leader) {
            prefetch_tensormap(&p.map_q);
            prefetch_tensormap(&p.map_k);
            prefetch_tensormap(&p.map_doh);
            prefetch_tensormap(&p.map_dol);
            prefetch_tensormap(&p.map_drh);
            prefetch_tensormap(&p.map_drl);
        }
        bool ok = true;
        int it = 0, kq_pending = -1, dor_pending = -1, s_pending = -1, d_pending = -1, t_pending = -1;
        auto load_tile = [&](uint64_t *bar, uint32_t off, const uint8_t *src, uint32_t bytes) {  // a whole operand tile
            if (leader) {
                mbar_arrive_expect_tx(bar, bytes);
                bulk_load(sm + off, src, bytes, bar);
            }
            __syncwarp();
        };
        // dO and -dR of item w into rows 0-63 / 64-127 of the [dO; -dR] tile (hi and lo)
        auto load_dor = [&](int w) {
            if (leader) {
                const Item I = item_of(p, w, nc);
                mbar_arrive_expect_tx(&bars->tma_dor, 4 * 16384);
                for (int cb = 0; cb < 2; ++cb) {
                    uint8_t *dor_cb = sm + OFF_DOR + cb * 16384;
                    tma_load_4d(dor_cb, &p.map_doh, &bars->tma_dor, cb * 64, I.h, I.t0, I.b);
                    tma_load_4d(dor_cb + LO_128, &p.map_dol, &bars->tma_dor, cb * 64, I.h, I.t0, I.b);
                    tma_load_4d(dor_cb + 8192, &p.map_drh, &bars->tma_dor, cb * 64, I.h, I.t0, I.b);
                    tma_load_4d(dor_cb + LO_128 + 8192, &p.map_drl, &bars->tma_dor, cb * 64, I.h, I.t0, I.b);
                }
            }
            __syncwarp();
        };

        auto wait = [&](uint64_t *bar, int parity) {
            ok = ok && wait_bar_warp(bar, parity, abort_flag, wait_ns);
            tc_fence_after();
            return ok;
        };
        if (p.debug_stall) ok = wait_bar_warp(&bars->never, 0, abort_flag, wait_ns);
        for (int w = blockIdx.x; w < p.items; w += gridDim.x, ++it) {
            const int ph = it & 1;
            if (!ok) break;
            const Item I = item_of(p, w, nc);
            // the previous item's last products are complete: every operand tile is free
            if (it > 0 && !wait(&bars->m2, ph ^ 1)) break;
            if (leader) {
                mbar_arrive_expect_tx(&bars->tma_kq, 2 * 16384);
                for (int cb = 0; cb < 2; ++cb) {
                    tma_load_4d(sm + OFF_KQ + cb * 16384, &p.map_k, &bars->tma_kq, cb * 64, I.h, I.t0, I.b);
                    tma_load_4d(sm + OFF_KQ + cb * 16384 + 8192, &p.map_q, &bars->tma_kq, cb * 64, I.h, I.t0, I.b);
                }
            }
            kq_pending = ph;
            __syncwarp();
            // queued behind K and Q (the Gram needs only those), in the order of their first use
            load_tile(&bars->s_full, OFF_SS, p.states + (size_t)w * 65536, 65536);
            s_pending = ph;
            load_tile(&bars->t_full, OFF_W, p.tpp + (size_t)w * 16384, 16384);
            t_pending = ph;
            load_dor(w);
            dor_pending = ph;
            if (!wait(&bars->tma_kq, ph)) break;
            kq_pending = -1;
            if (leader) {  // Gram K K^T (rows 64-127 of the M = 128 product are Q K^T, unused)
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_bf16(tmem + TM_U, smem_desc(kq + off, 16, 1024), smem_desc(kq + off, 16, 1024), idesc, ks > 0);
                }
                mma_commit(&bars->g);
            }
            __syncwarp();
            if (!wait(&bars->s_full, ph)) break;
            s_pending = -1;
            if (leader) {  // X^T = S^T K^T: S^T read as an MN-major A (M = j), K = i
                const uint32_t idesc = idesc_bf16_f32(128, 64, 1, 0);
#pragma unroll 1
                for (int part = 0; part < 2; ++part)
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t boff = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16(tmem + TM_X, smem_desc(ss + part * LO_128 + ks * 2048, 16384, 1024),
                                 smem_desc(kq + boff, 16, 1024), idesc, (part | ks) != 0);
                    }
                mma_commit(&bars->m1a);
            }
            __syncwarp();
            if (!wait(&bars->tma_dor, ph)) break;
            dor_pending = -1;
            if (it > 0 && !wait(&bars->w_free, ph ^ 1)) break;  // the previous dQ^T and dK^T are read out
            if (leader) {
                {  // [dQ^T | dK^T] = S [dO; -dR]^T: one N = 128 product, K = j
                    const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll 1
                    for (int pr = 0; pr < 3; ++pr) {  // S hi x hi, S hi x lo, S lo x hi
                        const uint32_t a_lo = pr == 2 ? LO_128 : 0, b_lo = pr == 1 ? LO_128 : 0;
#pragma unroll 1
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                            mma_bf16(tmem + TM_DQ, smem_desc(ss + a_lo + off, 16, 1024),
                                     smem_desc(dor + b_lo + off, 16, 1024), idesc, (pr | ks) != 0);
                        }
                    }
                }
                mma_commit(&bars->m1b);
            }
            __syncwarp();
            if (!wait(&bars->m1b, ph)) break;  // the S tile is read: dS' replaces it
            load_tile(&bars->d_full, OFF_SS, p.dse + (size_t)w * 65536, 65536);
            d_pending = ph;
            if (!wait(&bars->w_u, ph)) break;  // R^T split written, zero keys' T'' entries set (after t_full)
            if (leader) {  // U^T = R^T T''^T: A = R^T split (TMEM), B[t][s] = T''[t][s] (K-major)
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t bh = smem_desc(wt + ks * 32, 16, 1024), bl = smem_desc(wt + LO_64 + ks * 32, 16, 1024);
                    mma_bf16_ts(tmem + TM_U, tmem + TM_RS + ks * 8, bh, idesc, ks > 0);
                    mma_bf16_ts(tmem + TM_U, tmem + TM_RS + ks * 8, bl, idesc, 1);
                    mma_bf16_ts(tmem + TM_U, tmem + TM_RS + 32 + ks * 8, bh, idesc, 1);
                }
                mma_commit(&bars->u);
            }
            __syncwarp();
            if (!wait(&bars->w_p3, ph)) break;  // U^T split and tile, -G^T written
            if (!wait(&bars->d_full, ph)) break;
            d_pending = -1;
            if (leader) {
                {  // Z^T += U^T (-L)^T: A = U^T split (TMEM), B[t][s] = -L[t][s] (K-major)
                    const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t bh = smem_desc(l + ks * 32, 16, 1024), bl = smem_desc(l + LO_64 + ks * 32, 16, 1024);
                        mma_bf16_ts(tmem + TM_X, tmem + TM_US + ks * 8, bh, idesc, 1);
                        mma_bf16_ts(tmem + TM_X, tmem + TM_US + ks * 8, bl, idesc, 1);
                        mma_bf16_ts(tmem + TM_X, tmem + TM_US + 32 + ks * 8, bh, idesc, 1);
                    }
                }
                {  // -dY^T += (-dR)^T (-L): A[j][s] = -dR[s][j] (rows 64-127 of the [dO; -dR] tile, MN-major),
                   // B[t][s] = -L[s][t] (MN-major)
                    const uint32_t idesc = idesc_bf16_f32(128, 64, 1, 1);
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ah = smem_desc(dor + 8192 + ks * 2048, 16384, 1024);
                        const uint64_t al = smem_desc(dor + LO_128 + 8192 + ks * 2048, 16384, 1024);
                        const uint64_t bh = smem_desc(l + ks * 2048, 8192, 1024), bl = smem_desc(l + LO_64 + ks * 2048, 8192, 1024);
                        mma_bf16(tmem + TM_U, ah, bh, idesc, 1);
                        mma_bf16(tmem + TM_U, ah, bl, idesc, 1);
                        mma_bf16(tmem + TM_U, al, bh, idesc, 1);
                    }
                }
                mma_commit(&bars->a);
                // [dP; -dR U^T] = [dO; -dR] U^T, then dK^T += dS' U^T: B[t][j] = U^T[j][t] (MN-major), K = j
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
#pragma unroll 1
                for (int pr = 0; pr < 3; ++pr) {  // hi x hi, hi x lo, lo x hi
                    const uint32_t a_lo = pr == 2 ? LO_128 : 0, b_lo = pr == 1 ? LO_UT : 0;
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t aoff = a_lo + (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16(tmem + TM_P, smem_desc(dor + aoff, 16, 1024), smem_desc(ut + b_lo + ks * 2048, 8192, 1024),
                                 idesc, (pr | ks) != 0);
                    }
                }
                mma_commit(&bars->b);
#pragma unroll 1
                for (int pr = 0; pr < 3; ++pr) {
                    const uint32_t a_lo = pr == 2 ? LO_128 : 0, b_lo = pr == 1 ? LO_UT : 0;
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t aoff = a_lo + (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16(tmem + TM_DK, smem_desc(ss + aoff, 16, 1024), smem_desc(ut + b_lo + ks * 2048, 8192, 1024),
                                 idesc, 1);
                    }
                }
            }
            __syncwarp();
            if (!wait(&bars->w_p5, ph)) break;  // dP and E tiles written
            if (leader) {  // dQ^T += K^T dP^T;  dK^T += Q^T dP + K^T E
                const uint32_t id_kn = idesc_bf16_f32(128, 64, 1, 0), id_mn = idesc_bf16_f32(128, 64, 1, 1);
#pragma unroll 1
                for (int part = 0; part < 2; ++part)
#pragma unroll 1
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t kt = smem_desc(kq + ks * 2048, 16384, 1024);         // K^T (M = i, K = s)
                        const uint64_t qt = smem_desc(kq + 8192 + ks * 2048, 16384, 1024);  // Q^T
                        const uint32_t lo = part * LO_64;
                        mma_bf16(tmem + TM_DQ, kt, smem_desc(wt + lo + ks * 32, 16, 1024), id_kn, 1);      // dP[t][s]
                        mma_bf16(tmem + TM_DK, qt, smem_desc(wt + lo + ks * 2048, 8192, 1024), id_mn, 1);  // dP[s][t]
                        mma_bf16(tmem + TM_DK, kt, smem_desc(l + lo + ks * 32, 16, 1024), id_kn, 1);       // E[t][s]
                    }
                mma_commit(&bars->m2);
            }
            __syncwarp();
        }
        if (!ok) *abort_flag = 1;
        if (leader) {  // every product and load issued has completed before TMEM and the CTA go (bounded)
            mma_commit(&bars->drain);
            const uint64_t ts = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->drain, 0, 20000) && globaltimer_ns() - ts < DRAIN_NS) {
            }
            while (kq_pending >= 0 && !mbar_try_wait_sleep(&bars->tma_kq, kq_pending, 20000) &&
                   globaltimer_ns() - ts < DRAIN_NS) {
            }
            while (dor_pending >= 0 && !mbar_try_wait_sleep(&bars->tma_dor, dor_pending, 20000) &&
                   globaltimer_ns() - ts < DRAIN_NS) {
            }
            while (s_pending >= 0 && !mbar_try_wait_sleep(&bars->s_full, s_pending, 20000) &&
                   globaltimer_ns() - ts < DRAIN_NS) {
            }
            while (d_pending >= 0 && !mbar_try_wait_sleep(&bars->d_full, d_pending, 20000) &&
                   globaltimer_ns() - ts < DRAIN_NS) {
            }
            while (t_pending >= 0 && !mbar_try_wait_sleep(&bars->t_full, t_pending, 20000) &&
                   globaltimer_ns() - ts < DRAIN_NS) {
            }
        }
        __syncwarp();
    } else {
        // ============================ CUDA-core warps ============================
        float *row_dadb = reinterpret_cast<float *>(sm + OFF_ROW), *row_dadl = row_dadb + C, *row_dal = row_dadl + C;
        float *dLs = reinterpret_cast<float *>(sm + OFF_DOR);  // dL (P4)
        // TMEM: this thread reads and writes lane `ln` (its warp's quarter), the columns of token half `hf`
        const int hf = warp >> 2, ln = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const bool gate_thr = ln < C && (ln >> 5) == hf;  // holds K K^T[t][t] for t = ln
        bool ok = true;
        int it = 0;
        auto wait = [&](uint64_t *bar, int parity) {
            ok = ok && wait_bar_warp(bar, parity, abort_flag, wait_ns);
            tc_fence_after();
        };
        // operands of this warp written (generic and TMEM stores): one arrival per warp
        auto hand_over = [&](uint64_t *bar) {
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        for (int w = blockIdx.x; w < p.items; w += gridDim.x, ++it) {
            const int ph = it & 1;
            const Item I = item_of(p, w, nc);
            const int valid = I.valid;
            const size_t row0 = I.row0;
            const float bt = gate_thr && ln < valid ? p.beta[row0 + (size_t)ln * p.H] : 0.f;
            if (tid < C) row_dal[tid] = 0.f;  // (read by this thread only, in the previous item's dbeta)
            // ------------------------------ P0: gate terms, -L ------------------------------
            wait(&bars->g, ph);
            bool zero_key = false;  // this gate thread's key is zero: T''[t][t] = alpha_t (the forward has 0)
            float alpha = 0.f;
            if (ok && ln < C) {  // row t = ln of K K^T, this half's 32 columns (warps 0, 1, 4, 5)
                const int t = ln, col0 = 32 * hf;
                float g[32];
                tmem_ld32(lane_base + TM_U + col0, g);
                tmem_ld_wait();
                if (gate_thr) {
                    float lam = 0.f;
#pragma unroll
                    for (int s = 0; s < 32; ++s) lam = (s == (t & 31)) ? g[s] : lam;
                    float db = 0.f, dl = 0.f;
                    if (t < valid) gate_grad(bt, lam, p.euler, db, dl);
                    row_dadb[t] = db;
                    row_dadl[t] = dl;
                    zero_key = t < valid && !(lam > 0.f);
                    alpha = efla_alpha(bt, lam, p.euler);
                }
                float x[32];
#pragma unroll
                for (int s = 0; s < 32; ++s) x[s] = col0 + s < t ? -g[s] : 0.f;  // -L
                put16(sm + OFF_L, LO_64, t, col0, x);
                put16(sm + OFF_L, LO_64, t, col0 + 16, x + 16);
            }
            if (named_bar_any(BAR_W, NW, !ok)) break;  // every CUDA-core warp leaves together
            // ------------------------------ P2: R^T, dS' ------------------------------
            float gt[32];
            wait(&bars->m1a, ph);    // X^T complete
            wait(&bars->t_full, ph);  // the forward's T'' landed
            if (ok && zero_key) {     // u_t = alpha_t r_t for a zero key
                const uint32_t b = __float_as_uint(alpha), off = swz_offset(ln, ln, 0);
                const uint32_t lo = __float_as_uint(alpha - __uint_as_float(b & 0xffff0000u));
                *reinterpret_cast<uint16_t *>(sm + OFF_W + off) = (uint16_t)(b >> 16);
                *reinterpret_cast<uint16_t *>(sm + OFF_W + LO_64 + off) = (uint16_t)(lo >> 16);
            }
            if (ok) {
                // V^T: rows past the chunk's end load its last row (always in bounds) and are zeroed
                // after, so that all 32 loads are unconditional and in flight together
                const __nv_bfloat16 *vc = p.v + row0 * D + ln;
                __nv_bfloat16 vr[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) vr[e] = __ldcg(vc + (size_t)min(32 * hf + e, valid - 1) * p.H * D);
                // -G^T of this lane and token half (loads as for V^T), kept for P3
#pragma unroll
                for (int e = 0; e < 32; ++e) gt[e] = __ldcg(p.g + (row0 + (size_t)min(32 * hf + e, valid - 1) * p.H) * D + ln);
                float r[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = 32 * hf + e < valid ? __bfloat162float(vr[e]) : 0.f;
                float xt[32];
                tmem_ld32(lane_base + TM_X + 32 * hf, xt);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] -= xt[e];  // R^T = V^T - X^T
                tmem_st32(lane_base + TM_X + 32 * hf, r);
                tsplit32(lane_base, TM_RS, hf, r);
            }
            hand_over(&bars->w_u);
            // ------------------------------ P3 operands ------------------------------
            wait(&bars->u, ph);
            if (ok) {
#pragma unroll
                for (int e = 0; e < 32; ++e) gt[e] = 32 * hf + e < valid ? -gt[e] : 0.f;
                float u[32];
                tmem_ld32(lane_base + TM_U + 32 * hf, u);
                tmem_ld_wait();
                tsplit32(lane_base, TM_US, hf, u);
                put16(sm + OFF_UT, LO_UT, ln, 32 * hf, u);
                put16(sm + OFF_UT, LO_UT, ln, 32 * hf + 16, u + 16);
                tmem_st32(lane_base + TM_U + 32 * hf, gt);  // -G^T over U^T (read above)
            }
            hand_over(&bars->w_p3);
            // ------------------------------ P4 ------------------------------
            wait(&bars->a, ph);
            if (ok) {  // dalpha_t: sum over j of dY^T[j][t] Z^T[j][t]; this warp's 32 lanes, then across warps
                float y[32], z[32];
                tmem_ld32(lane_base + TM_U + 32 * hf, y);
                tmem_ld32(lane_base + TM_X + 32 * hf, z);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) y[e] *= -z[e];  // TM_U holds -dY^T
                atomicAdd(&row_dal[32 * hf + lane], lane_reduce_scatter(y, lane));
            }
            wait(&bars->b, ph);
            if (ok) {
                float x[32];
                tmem_ld32(lane_base + TM_P + 32 * hf, x);
                tmem_ld_wait();
                if (ln < C) {  // dP = (dO U^T) o M_incl, row t
                    const int t = ln;
#pragma unroll
                    for (int s = 0; s < 32; ++s) x[s] = 32 * hf + s <= t ? x[s] : 0.f;
                    put16(sm + OFF_W, LO_64, t, 32 * hf, x);
                    put16(sm + OFF_W, LO_64, t, 32 * hf + 16, x + 16);
                } else {  // dL = strictly-lower(-dR U^T), row t
                    const int t = ln - C;
#pragma unroll
                    for (int s = 0; s < 32; ++s) dLs[t * DL_LD + 32 * hf + s] = 32 * hf + s < t ? x[s] : 0.f;
                }
            }
            if (named_bar_any(BAR_W, NW, !ok)) break;
            {  // E = dL + dL^T + diag(2 dalpha dalpha/dlambda): the gate's share of dk rides on K^T E
                const int t = tid >> 2, s0 = (tid & 3) * 16;
                const float dg = 2.f * row_dal[t] * row_dadl[t];
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x[e] = dLs[t * DL_LD + s0 + e] + dLs[(s0 + e) * DL_LD + t] + (s0 + e == t ? dg : 0.f);
                put16(sm + OFF_L, LO_64, t, s0, x);
            }
            if (tid < valid) p.dbeta[row0 + (size_t)tid * p.H] = row_dal[tid] * row_dadb[tid];
            hand_over(&bars->w_p5);
            // ------------------------------ P6 ------------------------------
            wait(&bars->m2, ph);
            if (ok) {
                float dq[32], dk[32];
                tmem_ld32(lane_base + TM_DQ + 32 * hf, dq);
                tmem_ld32(lane_base + TM_DK + 32 * hf, dk);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->w_free);  // dQ^T and dK^T are in registers
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int t = 32 * hf + e;
                    if (t < valid) {
                        const size_t o = (row0 + (size_t)t * p.H) * D + ln;
                        p.dq[o] = dq[e];
                        p.dk[o] = dk[e];
                    }
                }
            }
        }
        if (!ok) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();  // every role is done: an abort flagged by any of them is visible now
    if (tid == 0 && *abort_flag) atomicExch(p.status, (int)EFLA_ERR_DEVICE_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

// Per-chunk gradients on the tensor cores: bf16 q, k, v, d_k = d_v = 128, T > 0, after
// launch_bwd_state_tc (dse, G in g, -dR split in dr_split, dO split in do_split) and the forward
// with chunk-start states and T'' tiles.  Persistent: one CTA per
// SM at most, each walking items blockIdx.x, blockIdx.x + gridDim.x, ...
cudaError_t launch_bwd_grad_tc(const BwdArgs &a, const float *states, const float *dse, const uint8_t *tpp,
                               const void *do_split, const float *g, const void *dr_split, const char **why) {
    const long items = (long)a.B * a.H * ((a.T + C - 1) / C);
    if (items == 0) return cudaSuccess;
    const size_t n = (size_t)a.B * a.T * a.H * D;
    const __nv_bfloat16 *hi = static_cast<const __nv_bfloat16 *>(do_split), *lo = hi + n;
    const __nv_bfloat16 *rhi = static_cast<const __nv_bfloat16 *>(dr_split), *rlo = rhi + n;
    GtParams p;
    memset(&p, 0, sizeof p);
    if (!bwd_row_map(&p.map_q, a.q, a.B, a.T, a.H) || !bwd_row_map(&p.map_k, a.k, a.B, a.T, a.H) ||
        !bwd_row_map(&p.map_doh, hi, a.B, a.T, a.H) || !bwd_row_map(&p.map_dol, lo, a.B, a.T, a.H) ||
        !bwd_row_map(&p.map_drh, rhi, a.B, a.T, a.H) || !bwd_row_map(&p.map_drl, rlo, a.B, a.T, a.H)) {
        *why = "cuTensorMapEncodeTiled failed";
        return cudaErrorInvalidValue;
    }
    p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.beta = a.beta;
    p.states = reinterpret_cast<const uint8_t *>(states);
    p.dse = reinterpret_cast<const uint8_t *>(dse);
    p.tpp = tpp;
    p.g = g;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dbeta = a.dbeta;
    p.status = device_status_ptr();
    p.T = a.T;
    p.H = a.H;
    p.items = (int)items;
    p.euler = a.euler;
    p.wait_ns = wait_limit_ns();
    p.debug_stall = (debug_stall() & STALL_BWD_GRAD) ? 1 : 0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        *why = "querying the SM count";
        return e;
    }
    static bool attr_done[64] = {};
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(bwd_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
        if (e != cudaSuccess) {
            *why = "setting the gradient kernel's shared memory";
            return e;
        }
        if (dev < 64) attr_done[dev] = true;
    }
    *why = "tcgen05 gradient kernel launch";
    bwd_grad_tc_kernel<<<(unsigned)std::min<long>(items, sms), NTH, SMEM_ALLOC, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace efla
