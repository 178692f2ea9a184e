// Chunkwise EFLA forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The recurrence S_t = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T,
// o_t = S_t^T q_t ("Exact Flow Linear Attention" (gist.science), Metodologia 3;
// "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-4) is
// evaluated in chunks of C = 64 tokens with the WY/UT representation of the
// product of the chunk's rank-1 updates.  For one chunk with start state S
// (d_k x d_v, fp32), keys K, queries Q, values V (C x d), and per row
//   lambda_t = ||k_t||^2,  n_t = sqrt(lambda_t),  gamma_t = 1 - e^{-beta_t lambda_t}
//   (gamma_t = alpha_t lambda_t, computed as -expm1(-beta_t lambda_t)):
//
//   A~  = strictly-lower( gamma_t (k_t . k_s) / (n_t n_s) )        (C x C)
//   T~  = (I + A~)^{-1}                                            (blocked forward substitution)
//   T'  = T~ diag(gamma / n)
//   U^  = T' (V - K S)            u_t = U^_t / n_t   (= the rank-1 write u_t of token t)
//   so u = T'' (V - K S) with T'' = diag(1/n) T~ diag(gamma / n).
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
// that the state's d_v index is the MMA row (TMEM lane) and the operands S^T,
// (V - X)^T and u^T are written into TMEM by the thread that owns the lane and
// read from there by the tensor core:
//   [X^T | O1^T] = S^T [K; Q]^T               (M = d_v = 128, N = 2C, K = d_k)
//   u^T  = V^T T''^T + (-X)^T T''^T           (M = 128, N = C, K = C; V^T read from
//                                              the stage as an MN-major operand)
//   O^T         += u^T P^T,  P = Q K^T o M   (M = 128, N = C, K = C)
//   S^T         += u^T K             (M = 128, N = d_k = 128, K = C; K as MN-major operand)
// and G = [K ; Q] K^T (M = 2C = 128, N = C, K = d_k) gives the chunk's Gram terms.
//
// One CTA of 448 threads per (sequence, head):
//   state warpgroup (threads 0-127): thread j owns TMEM lane j (column j of S);
//     runs the per-chunk dependency chain above and writes o with TMA stores.
//   MMA thread (warp 8): issues the state chain's tensor-core products.
//   TMA producer (warp 9): loads K, Q, V into three stages.
//   prep warpgroups (warps 4-7 and 10-13): form the Gram products, the gate terms,
//     T'' and P for the NEXT chunk while the state warpgroup works on the current one.
// Every wait is bounded; on expiry the CTA records EFLA_ERR_DEVICE_TIMEOUT and
// leaves.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tri_inverse.cuh"

namespace efla {
namespace {
using namespace ptx;
using namespace tc;

constexpr int C = 64;
constexpr int D = 128;

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr int NSTAGE = 3;
constexpr uint32_t STAGE_BYTES = 49152;    // [K;Q] [2 cb][128 rows][64] (32 KB) + V [2 cb][64 rows][64] (16 KB)
constexpr uint32_t OFF_STAGE = 0;          // NSTAGE stages
constexpr uint32_t OFF_V = 32768;          // within a stage
// Per chunk parity: T'' {hi 8 KB, lo 8 KB} [64 t][64 s], then P {hi, lo} [64 t][64 s].
// Once a chunk's last product has read them, the 32 KB hold that chunk's o tile
// on its way to the TMA store (4 warps x [64 t][32] fp32).
constexpr uint32_t OFF_TPP = NSTAGE * STAGE_BYTES;
constexpr uint32_t TPP_BYTES = 32768;
constexpr uint32_t OFF_AT = OFF_TPP + 2 * TPP_BYTES;  // fp32 [64][68]: A~, then T~ in place (rows 16-byte aligned)
constexpr uint32_t AT_LD = 68;
constexpr uint32_t OFF_ROW = OFF_AT + 64 * AT_LD * 4;  // fp32: invn[64], gn[64]
constexpr uint32_t ROW_BYTES = 2 * 64 * 4;
constexpr uint32_t OFF_BAR = OFF_ROW + ROW_BYTES;       // mbarriers (struct Bars)
constexpr uint32_t OFF_MISC = OFF_BAR + 224;            // tmem base (u32), abort flag (i32), sequence slot (i32)
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;       // + alignment slack for the 1024-byte base
static_assert(OFF_TPP % 1024 == 0 && OFF_AT % 1024 == 0, "operand buffers must be 1024-byte aligned");
static_assert(SMEM_ALLOC <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

// TMEM columns (32-bit; lane = row of the MMA result)
// A tcgen05.mma of M = 128 occupies the tensor pipe for about the same time at
// N = 64 as at N = 128, so products that share their A operand are issued as one
// instruction over adjacent B rows and adjacent accumulator columns.
constexpr uint32_t TM_S = 0;    // S^T fp32                                       128 columns
constexpr uint32_t TM_SA = 128; // S^T as bf16 operand: hi 64, lo 64; then the two
                                // partial sums of u^T (fp32, 64 + 64)
constexpr uint32_t TM_X = 256;  // X^T fp32 (64), then (-X)^T bf16 hi 32 + lo 32, then u^T bf16 hi 32 + lo 32
constexpr uint32_t TM_O = 320;  // O^T fp32 of even chunks (64); odd chunks at TM_O + 64
constexpr uint32_t TM_G = 448;  // [K;Q] K^T fp32                                  64 columns
constexpr uint32_t TM_COLS = 512;

// Bound on the waits that let a CTA's own copies and tensor-core operations finish before it
// releases tensor memory.  The waits between roles are bounded by TcParams::wait_ns.
constexpr uint64_t WAIT_NS = 2000000000ull;

constexpr int BAR_PREP = 2;
// Packed batches of at most this many sequences are run longest first (each CTA ranks the
// sequence lengths itself: N^2 / threads comparisons).
constexpr int LONGEST_FIRST_MAX_N = 128;  // named barrier of the two prep warpgroups (256 threads)

struct TcParams {
    CUtensorMap map_q;
    CUtensorMap map_k;
    CUtensorMap map_v;
    CUtensorMap map_o;
    const float *beta;
    const float *S0;
    const int32_t *cu_seqlens;
    void *o;
    float *S_T;
    int *status;
    int B, T, H, N;
    int euler;  // 1: delta-rule gate (gamma = beta * lambda)
    // Sequences split into segments (seg_len > 0; rows of [B, T] only, no cu_seqlens):
    //   map launch (maps != nullptr): CTAs (pass, b, g < G-1, h); pass 0 runs segment g from
    //     S = I with v = 0, pass 1 from S = 0; neither writes o; S_T goes to maps[pass][b][g][h].
    //   output launch: CTAs (b, g, h) start from s_in[b][g][h]; only g = G-1 writes S_T[b][h].
    int seg_len, G;
    const float *s_in;
    float *maps;
    float *states;               // chunk-start states [N, H, nchunks] x 64 KB (rows of [B, T]) or nullptr: S as
                                 // bf16 hi/lo operand tiles (put_col_split_tile) for the tensor-core backward
    uint8_t *tpp;                // with states: every chunk's T'' tile as formed below (16 KB a chunk) or nullptr
    unsigned long long wait_ns;  // bound on every wait between roles (2 s unless a test lowers it)
    int debug_stall;             // test hook: the MMA thread first waits on a barrier nothing completes
};

struct Bars {
    uint64_t tma_full[NSTAGE];  // K, Q, V of a stage landed
    uint64_t g_done;         // Gram MMA of a chunk complete
    uint64_t g_free;         // the prep warpgroups have read a chunk's Gram products
    uint64_t x_done;         // X^T = S^T K^T
    uint64_t u_done;         // U^^T
    uint64_t s_done;         // S^T += u^T K
    uint64_t prep_ready[2];  // T', P, gate terms and the zeroed tail of a chunk written
    uint64_t sa_ready;       // state warpgroup wrote S^T hi/lo        (128 arrivals)
    uint64_t r_ready;        // state warpgroup wrote (V - X)^T hi/lo  (128 arrivals)
    uint64_t u_ready;        // state warpgroup wrote u^T hi/lo        (128 arrivals)
    uint64_t drain[2];       // all MMAs of the MMA thread / of the prep thread complete
    uint64_t s_free[NSTAGE];  // the state update of a chunk complete: its K/Q/V stage is free
    // Per chunk parity b (chunk c uses O^T buffer c & 1 and T''/P buffer c & 1):
    uint64_t o_done[2];       // the chunk's O^T products complete (its P part is free again)
    uint64_t o_free[2];       // the state warpgroup has read the chunk's O^T  (128 arrivals)
    uint64_t stg_free[2];     // the TMA stores of the chunk's o tile have read their staging,
                              // the T'' part of its buffer (4 arrivals)
    uint64_t never;           // never completed (the debug_stall test hook waits on it)
};
static_assert(sizeof(Bars) <= 224, "mbarrier block exceeds its slot");

// G = [K; Q] K^T of chunk c (M = 128, N = C, K = d_k) into TM_G, completion on g_done.
__device__ __forceinline__ void issue_gram(uint32_t tmem, uint32_t s_sm, int c, Bars *bars) {
    const uint32_t kq = s_sm + OFF_STAGE + (c % NSTAGE) * STAGE_BYTES;
    const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tmem + TM_G, smem_desc(kq + off, 16, 1024), smem_desc(kq + off, 16, 1024), idesc, ks > 0);
    }
    mma_commit(&bars->g_done);
}

// Rows 32 g0 .. 32 g0 + 63 of the state S (column j = this thread's TMEM lane, TMEM address
// ts of S^T) into the backward's operand tile.  Out of line: only the forward that keeps its
// chunk states calls it, and the per-chunk loop's code stays small for the instruction cache.
__device__ __noinline__ void dump_state_rows(uint8_t *tile, uint32_t ts, int g0, int j) {
#pragma unroll 1
    for (int g = g0; g < g0 + 2; ++g) {
        float sv[32];
        tmem_ld32(ts + g * 32, sv);
        tmem_ld_wait();
        put_col_split_tile(tile, g * 32, j, sv);
    }
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(448, 1) chunk_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *row_invn = reinterpret_cast<float *>(sm + OFF_ROW);  // [64] 1/n_t
    float *row_gn = row_invn + 64;                              // [64] gamma_t/n_t
    float *At = reinterpret_cast<float *>(sm + OFF_AT);
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint64_t wait_ns = p.wait_ns;
    long b, bos, eos;
    int h;
    int mode = 0;                    // 0: forward; 1: map from S = I, v = 0; 2: map from S = 0
    const float *s0p = nullptr;      // this CTA's start state (nullptr: zero)
    float *stp = nullptr;            // where this CTA's final state goes (nullptr: nowhere)
    if (p.seg_len > 0) {  // a segment of a split sequence
        int idx = blockIdx.x;
        const int Gu = p.maps ? p.G - 1 : p.G;
        if (p.maps) {
            const int per_pass = p.B * Gu * p.H;
            mode = 1 + idx / per_pass;
            idx %= per_pass;
        }
        h = idx % p.H;
        idx /= p.H;
        const int g = idx % Gu;
        b = idx / Gu;
        bos = (long)g * p.seg_len;
        eos = min((long)p.T, bos + p.seg_len);
        if (mode == 0) {
            s0p = p.s_in + (((size_t)b * p.G + g) * p.H + h) * D * D;
            if (g == p.G - 1 && p.S_T) stp = p.S_T + ((size_t)b * p.H + h) * D * D;
        } else {
            stp = p.maps + ((((size_t)(mode - 1) * p.B + b) * Gu + g) * p.H + h) * D * D;
        }
    } else {
        int n = blockIdx.x / p.H;
        h = blockIdx.x % p.H;
        if (p.cu_seqlens && p.N <= LONGEST_FIRST_MAX_N) {
            // Longest first: the CTAs of group r (blockIdx / H = r, dispatched roughly in that
            // order) run the r-th longest sequence (ties by index), so the long sequences start
            // early and the short ones fill the tail.  The ranks are a permutation of 0..N-1.
            int *len = reinterpret_cast<int *>(sm + OFF_AT);  // free until the prep starts
            int *slot = reinterpret_cast<int *>(sm + OFF_MISC + 8);
            if (tid < p.N) len[tid] = p.cu_seqlens[tid + 1] - p.cu_seqlens[tid];
            __syncthreads();
            if (tid < p.N) {
                const int li = len[tid];
                int rank = 0;
                for (int j = 0; j < p.N; ++j) rank += (len[j] > li) || (len[j] == li && j < tid);
                if (rank == n) *slot = tid;
            }
            __syncthreads();
            n = *slot;
            __syncthreads();  // every thread has read the slot before the scratch is reused
        }
        if (p.cu_seqlens) {
            b = 0;
            bos = p.cu_seqlens[n];
            eos = p.cu_seqlens[n + 1];
            if (bos < 0 || eos < bos || eos > p.T) {  // malformed bounds: flag and touch nothing
                if (tid == 0) atomicExch(p.status, (int)EFLA_ERR_INVALID_ARG);
                return;
            }
        } else {
            b = n;
            bos = 0;
            eos = p.T;
        }
        const size_t sbase = ((size_t)n * p.H + h) * D * D;
        if (p.S0) s0p = p.S0 + sbase;
        if (p.S_T) stp = p.S_T + sbase;
    }
    const bool write_o = mode == 0 && p.o != nullptr;
    const int nchunks = eos > bos ? (int)((eos - bos + C - 1) / C) : 0;

    if (nchunks == 0) {  // empty sequence: S_T = S0
        if (stp && tid < D)
            for (int i = 0; i < D; ++i)
                stp[(size_t)i * D + tid] = mode == 1 ? (i == tid ? 1.f : 0.f) : s0p ? s0p[(size_t)i * D + tid] : 0.f;
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&bars->tma_full[i], 1);
            mbar_init(&bars->s_free[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->o_done[i], 1);
            mbar_init(&bars->o_free[i], 128);
            mbar_init(&bars->stg_free[i], 4);
            mbar_init(&bars->prep_ready[i], 1);
            mbar_init(&bars->drain[i], 1);
        }
        mbar_init(&bars->g_done, 1);
        mbar_init(&bars->g_free, 1);
        mbar_init(&bars->x_done, 1);
        mbar_init(&bars->u_done, 1);
        mbar_init(&bars->s_done, 1);
        mbar_init(&bars->sa_ready, 128);
        mbar_init(&bars->r_ready, 128);
        mbar_init(&bars->u_ready, 128);
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
    const uint32_t s_sm = smem_u32(sm);

    if ((tid >= 128 && tid < 256) || tid >= 320) {
        // ============================== prep warpgroups ==============================
        // Warps 4-7 and 10-13 share each chunk's CUDA-core work (256 threads, index pi).
        // Gram row r (TMEM lane r) is read by one thread of each warpgroup: columns
        // 0-31 by warps 4-7, columns 32-63 by warps 10-13.
        const int half = tid >= 320 ? 1 : 0;
        const int pi = half ? tid - 320 + 128 : tid - 128;
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row = quarter * 32 + (tid & 31);
        const int col0 = half * 32;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool leader = pi == 0;  // signals the other roles
        // The thread that reads the Gram diagonal of row t computes that row's gate terms;
        // it loads beta_t itself, a chunk ahead (its latency hides behind the prep).
        const bool gate_thr = row < C && (row >> 5) == half;
        auto load_beta = [&](int cc) {
            const long t0n = bos + (long)cc * C;
            return (cc < nchunks && gate_thr && t0n + row < eos)
                       ? p.beta[((size_t)b * p.T + (size_t)(t0n + row)) * p.H + h] : 0.f;
        };
        float beta_next = load_beta(0);
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % NSTAGE, buf = c & 1;
            const long tok0 = bos + (long)c * C;
            const int valid = (int)min((long)C, eos - tok0);
            uint8_t *KQ = sm + OFF_STAGE + st * STAGE_BYTES;

            const float beta_t = beta_next;
            beta_next = load_beta(c + 1);
            bool ok = true;
            // Gram products G = [K;Q] K^T: the MMA thread issues a full chunk's once its stage
            // has landed (the prep reads nothing else of the stage); a partial chunk's tail is
            // zeroed here first (those rows may hold the next sequence) and its product issued
            // by the prep
            if (valid < C) {
                ok = wait_bar(&bars->tma_full[st], (c / NSTAGE) & 1, abort_flag, wait_ns);
                if (ok) {
                    const int rows = C - valid;
                    for (int e = pi; e < 4 * rows * 8; e += 256) {
                        const int ch = e & 7, r = (e >> 3) % rows, part = (e >> 3) / rows;
                        const int R = valid + r + ((part >> 1) ? 64 : 0), cb = part & 1;
                        *reinterpret_cast<uint4 *>(KQ + cb * 16384 + (R >> 3) * 1024 + (R & 7) * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                if (named_bar_any(BAR_PREP, 256, !ok || *abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                if (leader) {
                    tc_fence_after();
                    issue_gram(tmem, s_sm, c, bars);
                }
            }
            ok = wait_bar_warp(&bars->g_done, c & 1, abort_flag, wait_ns);
            // This chunk's T''/P buffer was last read by chunk c-2: its P part by that chunk's
            // O^T products (o_done), its T'' part by the stores of that chunk's o tile (stg_free,
            // waited before T'' is written below).
            if (c >= 2) ok = wait_bar_warp(&bars->o_done[c & 1], ((c - 2) >> 1) & 1, abort_flag, wait_ns) && ok;
            tc_fence_after();
            {
                float g[32];
                tmem_ld32(lane_base + TM_G + col0, g);
                tmem_ld_wait();
                tc_fence_before();  // the next Gram MMA may overwrite TM_G once every row is read
                // [gate: G row loaded]
                if (row < C && (row >> 5) == half) {  // this thread holds K K^T[t][t]: gate terms of row t
                    const int t = row;
                    float lam = 0.f;
#pragma unroll
                    for (int s = 0; s < 32; ++s) lam = (s == (t & 31)) ? g[s] : lam;
                    const bool live = t < valid && lam > 0.f;
                    const float invn = live ? rsqrtf(lam) : 0.f;
                    const float gam = !live ? 0.f : p.euler ? beta_t * lam : -expm1f(-beta_t * lam);
                    row_invn[t] = invn;
                    row_gn[t] = gam * invn;
                }
                // [gate: terms computed]
                if (named_bar_any(BAR_PREP, 256, !ok || *abort_flag)) {  // also spreads an abort
                    *abort_flag = 1;
                    break;
                }
                // [gate: barrier passed]
                if (leader) mbar_arrive(&bars->g_free);  // every row of G has been read
                if (row < C) {  // A~[t][col0 .. col0+31]
                    const int t = row;
                    const float rs = row_gn[t];  // gamma_t / n_t
                    float iv[32];  // all scales first: the stores below may alias them for the compiler
#pragma unroll
                    for (int s4 = 0; s4 < 8; ++s4) {
                        const float4 f = reinterpret_cast<const float4 *>(row_invn + col0)[s4];
                        iv[4 * s4] = f.x;
                        iv[4 * s4 + 1] = f.y;
                        iv[4 * s4 + 2] = f.z;
                        iv[4 * s4 + 3] = f.w;
                    }
                    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
                    for (int s4 = 0; s4 < 32; s4 += 4) {  // (rs iv) g, two columns per packed fp32x2 multiply
                        const float2 a = __fmul2_rn(__fmul2_rn(rs2, make_float2(iv[s4], iv[s4 + 1])),
                                                    make_float2(g[s4], g[s4 + 1]));
                        const float2 c = __fmul2_rn(__fmul2_rn(rs2, make_float2(iv[s4 + 2], iv[s4 + 3])),
                                                    make_float2(g[s4 + 2], g[s4 + 3]));
                        float4 w;
                        w.x = col0 + s4 + 0 < t ? a.x : 0.f;
                        w.y = col0 + s4 + 1 < t ? a.y : 0.f;
                        w.z = col0 + s4 + 2 < t ? c.x : 0.f;
                        w.w = col0 + s4 + 3 < t ? c.y : 0.f;
                        *reinterpret_cast<float4 *>(At + t * AT_LD + col0 + s4) = w;
                    }
                } else if (write_o) {  // P[t][col0 .. col0+31] = Q K^T with the inclusive causal mask
                    const int t = row - C;
#pragma unroll
                    for (int s = 0; s < 32; ++s) g[s] = col0 + s <= t ? g[s] : 0.f;
                    uint8_t *phi = sm + OFF_TPP + buf * TPP_BYTES + 16384, *plo = phi + 8192;
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        uint32_t hh[4], ll[4];
                        split_pack<4>(g + c8, hh, ll);
                        const uint32_t off = swz_offset(t, col0 + c8, 8192);
                        *reinterpret_cast<uint4 *>(phi + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        *reinterpret_cast<uint4 *>(plo + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    }
                }
            }
            named_bar(BAR_PREP, 256);
            invert_unit_lower<BAR_PREP, AT_LD>(At, pi);
            if (c >= 2) ok = wait_bar_warp(&bars->stg_free[c & 1], ((c - 2) >> 1) & 1, abort_flag, wait_ns) && ok;
            {  // T'' = diag(1/n) T~ diag(gamma/n), lower triangle, as bf16 hi/lo [t][s]
                const int t = pi >> 2, s0 = (pi & 3) * 16;
                uint8_t *hi = sm + OFF_TPP + buf * TPP_BYTES, *lo = hi + 8192;
                // the same tile for the backward (a zero key's diagonal is 0 here; the backward sets it)
                uint8_t *ghi = p.tpp ? p.tpp + ((size_t)blockIdx.x * nchunks + c) * 16384 : nullptr;
                const float rsc = row_invn[t];
#pragma unroll
                for (int c8 = 0; c8 < 16; c8 += 8) {
                    float tt8[8], gn8[8];
                    *reinterpret_cast<float4 *>(tt8) = *reinterpret_cast<const float4 *>(At + t * AT_LD + s0 + c8);
                    *reinterpret_cast<float4 *>(tt8 + 4) = *reinterpret_cast<const float4 *>(At + t * AT_LD + s0 + c8 + 4);
                    *reinterpret_cast<float4 *>(gn8) = *reinterpret_cast<const float4 *>(row_gn + s0 + c8);
                    *reinterpret_cast<float4 *>(gn8 + 4) = *reinterpret_cast<const float4 *>(row_gn + s0 + c8 + 4);
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {  // (rsc T~) (gamma/n), two columns per packed multiply
                        const float2 y = __fmul2_rn(__fmul2_rn(make_float2(rsc, rsc), make_float2(tt8[e], tt8[e + 1])),
                                                    make_float2(gn8[e], gn8[e + 1]));
                        x[e] = s0 + c8 + e <= t ? y.x : 0.f;
                        x[e + 1] = s0 + c8 + e + 1 <= t ? y.y : 0.f;
                    }
                    uint32_t hh[4], ll[4];
                    split_pack<4>(x, hh, ll);
                    const uint32_t off = swz_offset(t, s0 + c8, 8192);
                    *reinterpret_cast<uint4 *>(hi + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                    *reinterpret_cast<uint4 *>(lo + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    if (ghi) {
                        *reinterpret_cast<uint4 *>(ghi + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        *reinterpret_cast<uint4 *>(ghi + 8192 + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            named_bar(BAR_PREP, 256);
            if (leader) mbar_arrive(&bars->prep_ready[buf]);
            if (!ok) *abort_flag = 1;  // seen by every prep thread at the next chunk's gate barrier
        }
        if (leader) {  // every Gram MMA has completed before TMEM is released (bounded)
            mma_commit(&bars->drain[1]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->drain[1], 0, 20000) && globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
    } else if (tid < 128) {
        // =============================== state warpgroup ===============================
        // Per chunk c, the dependency chain through the state is
        //   S -> X = K S -> V - X -> U^ -> u -> S + K^T u;
        // this warpgroup forms the operands of each link in TMEM and the MMA warp
        // issues the products.  The outputs of chunk c - 1 are read out and sent while the
        // tensor core updates the state of chunk c (off the chain).
        const int j = tid, lane = tid & 31;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        {  // initial state -> TMEM (S^T: lane j holds column j of S)
            float r[32];
#pragma unroll 1
            for (int g = 0; g < 4; g = opaque(g + 1)) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = mode == 1 ? (g * 32 + i == j ? 1.f : 0.f) : s0p ? s0p[(size_t)(g * 32 + i) * D + j] : 0.f;
                tmem_st32(lane_base + TM_S + g * 32, r);
            }
            tmem_st_wait();
        }
        // O^T of chunk cc (fp32 in TMEM buffer cc & 1) -> o.  Each warp stages its own 32
        // columns in its 4 KB slice of the T'' part of buffer cc & 1 (free: the chunk's u
        // products have read T'') and its lane 0 sends them with TMA stores, so no
        // cross-warp synchronisation is needed.  A bf16 tile (64 tokens x 32 columns) leaves
        // in one store, an fp32 tile in two halves of 32 tokens.  A partial chunk of a packed
        // batch is written with plain stores instead (a TMA box would spill into the next
        // sequence).  The staging is released later (release_staging), once the stores have
        // read it.
        auto epilogue = [&](int cc) {
            const uint32_t ob = TM_O + (uint32_t)(cc & 1) * 64;
            if (!write_o) {  // map modes: nothing to store
                tc_fence_before();
                mbar_arrive(&bars->o_free[cc & 1]);
                return;
            }
            const long t0c = bos + (long)cc * C;
            const int vc = (int)min((long)C, eos - t0c);
            float ov[32], ow[32];
            tmem_ld32(lane_base + ob, ov);
            tmem_ld32(lane_base + ob + 32, ow);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bars->o_free[cc & 1]);  // chunk cc + 2's first product may overwrite this O^T
            uint8_t *slice = sm + OFF_TPP + (cc & 1) * TPP_BYTES + warp * 4096;
            const bool full = p.cu_seqlens == nullptr || vc == C;
            auto store_rows = [&](int t_off, int n) {  // plain stores of staged rows (partial packed chunk)
#pragma unroll 1
                for (int t = 0; t < n; t = opaque(t + 1)) {
                    const size_t rw = ((size_t)b * p.T + (size_t)(t0c + t_off + t)) * p.H + h;
                    if (OUT_BF16)
                        static_cast<__nv_bfloat16 *>(p.o)[rw * D + j] =
                            reinterpret_cast<const __nv_bfloat16 *>(slice)[(t_off + t) * 32 + lane];
                    else
                        static_cast<float *>(p.o)[rw * D + j] = reinterpret_cast<const float *>(slice)[t * 32 + lane];
                }
            };
            if (OUT_BF16) {
                __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(slice) + lane;
#pragma unroll
                for (int t = 0; t < 32; ++t) stg[t * 32] = __float2bfloat16_rn(ov[t]);
#pragma unroll
                for (int t = 0; t < 32; ++t) stg[(32 + t) * 32] = __float2bfloat16_rn(ow[t]);
                if (full) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&p.map_o, slice, warp * 32, h, (int)t0c, (int)b);
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
                    store_rows(0, vc);
                    __syncwarp();
                }
            } else {
                auto send_half = [&](const float (&x)[32], int t_off) {
                    if (t_off > 0) {  // the first half's store has read the slice
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
                    }
                    float *stg = reinterpret_cast<float *>(slice) + lane;
#pragma unroll
                    for (int t = 0; t < 32; ++t) stg[t * 32] = x[t];
                    if (full) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_4d(&p.map_o, slice, warp * 32, h, (int)(t0c + t_off), (int)b);
                            bulk_commit();
                        }
                    } else {
                        __syncwarp();
                        store_rows(t_off, min(32, vc - t_off));
                        __syncwarp();
                    }
                };
                send_half(ov, 0);
                if (vc > 32) send_half(ow, 32);
            }
        };
        // The stores of chunk cc's o tile have read the staging: the prep of chunk cc + 2 may
        // write its T'' there.
        auto release_staging = [&](int cc) {
            if (lane == 0) {
                bulk_wait_read0();
                mbar_arrive(&bars->stg_free[cc & 1]);
            }
            __syncwarp();
        };
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            // The S^T operand needs only the previous state update, not this chunk's prep.
            if (c > 0) ok = wait_bar_warp(&bars->s_done, (c - 1) & 1, abort_flag, wait_ns);
            if (!ok) break;
            tc_fence_after();
            // S^T -> bf16 hi/lo operand in TMEM, 32 columns of S^T (16 operand columns) at a time;
            // with `states`, also the chunk's start state S (column j from this thread) as a bf16
            // hi/lo operand tile of the backward
            uint8_t *st_c = p.states ? reinterpret_cast<uint8_t *>(p.states + ((size_t)blockIdx.x * nchunks + c) * D * D)
                                     : nullptr;
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
            // with `states`, rows 0-63 of the start state go out while the tensor core forms X and
            // rows 64-127 while it forms u (TM_S changes only at this chunk's state update)
            if (st_c) dump_state_rows(st_c, lane_base + TM_S, 0, j);
            if (c >= 2) release_staging(c - 2);  // its stores were issued during chunk c - 1
            const long tok0 = bos + (long)c * C;
            const int valid = (int)min((long)C, eos - tok0);
            ok = wait_bar_warp(&bars->x_done, c & 1, abort_flag, wait_ns);
            if (!ok) break;
            tc_fence_after();
            // (-X)^T = -(K S)^T -> bf16 hi/lo operand in TMEM (rows past the sequence end are zero),
            // written over X once all of X is in registers
            {
                float x0[32], x1[32];
                tmem_ld32(lane_base + TM_X, x0);
                tmem_ld32(lane_base + TM_X + 32, x1);
                tmem_ld_wait();
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int t = 0; t < 32; ++t) x0[t] = t < valid ? -x0[t] : 0.f;
                split_pack<16>(x0, hi, lo);
                tmem_st16u(lane_base + TM_X, hi);
                tmem_st16u(lane_base + TM_X + 32, lo);
#pragma unroll
                for (int t = 0; t < 32; ++t) x1[t] = 32 + t < valid ? -x1[t] : 0.f;
                split_pack<16>(x1, hi, lo);
                tmem_st16u(lane_base + TM_X + 16, hi);
                tmem_st16u(lane_base + TM_X + 48, lo);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->r_ready);
            if (st_c) dump_state_rows(st_c, lane_base + TM_S, 2, j);
            ok = wait_bar_warp(&bars->u_done, c & 1, abort_flag, wait_ns);
            if (!ok) break;
            tc_fence_after();
            // u^T = U1 + U2 -> bf16 hi/lo operand in TMEM
#pragma unroll 1
            for (int hf = 0; hf < 2; hf = opaque(hf + 1)) {
                float u[32], u2[32];
                uint32_t hi[16], lo[16];
                tmem_ld32(lane_base + TM_SA + hf * 32, u);
                tmem_ld32(lane_base + TM_SA + 64 + hf * 32, u2);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; ++t) u[t] += u2[t];
                split_pack<16>(u, hi, lo);
                tmem_st16u(lane_base + TM_X + hf * 16, hi);
                tmem_st16u(lane_base + TM_X + 32 + hf * 16, lo);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->u_ready);
            // the outputs of the previous chunk leave while the tensor core updates the state
            if (c >= 1) {
                ok = wait_bar_warp(&bars->o_done[(c - 1) & 1], ((c - 1) >> 1) & 1, abort_flag, wait_ns);
                if (!ok) break;
                tc_fence_after();
                epilogue(c - 1);
            }
        }
        if (ok && nchunks >= 1) {  // the last chunk's outputs (its o_done also covers the last state update)
            ok = wait_bar_warp(&bars->o_done[(nchunks - 1) & 1], ((nchunks - 1) >> 1) & 1, abort_flag, wait_ns);
            if (ok) {
                tc_fence_after();
                epilogue(nchunks - 1);
            }
        }
        if (!ok) *abort_flag = 1;
        if (ok && stp) {  // final state
#pragma unroll 1
            for (int g = 0; g < 4; g = opaque(g + 1)) {
                float s32[32];
                tmem_ld32(lane_base + TM_S + g * 32, s32);
                tmem_ld_wait();
                float *dst = stp + (size_t)(g * 32) * D + j;
#pragma unroll
                for (int i = 0; i < 32; ++i) dst[(size_t)i * D] = s32[i];
            }
        }
        if (lane == 0) bulk_wait0();  // TMA stores have completed before the CTA leaves
    } else if (tid == 288) {
        // ============================ TMA producer (one thread) ============================
        // Chunk c goes into stage c % NSTAGE once the state update of chunk c - NSTAGE
        // (the last reader of that stage) has completed.
        prefetch_tensormap(&p.map_q);
        prefetch_tensormap(&p.map_k);
        prefetch_tensormap(&p.map_v);
        int issued = 0;
        for (int c = 0; c < nchunks; ++c) {
            if (c >= NSTAGE && !wait_bar(&bars->s_free[c % NSTAGE], ((c - NSTAGE) / NSTAGE) & 1, abort_flag, wait_ns)) break;
            const int st = c % NSTAGE;
            uint8_t *dst = sm + OFF_STAGE + st * STAGE_BYTES;
            const int tok = (int)(bos + (long)c * C);
            mbar_arrive_expect_tx(&bars->tma_full[st], STAGE_BYTES);
            for (int cb = 0; cb < 2; ++cb) {
                tma_load_4d(dst + cb * 16384, &p.map_k, &bars->tma_full[st], cb * 64, h, tok, (int)b);
                tma_load_4d(dst + cb * 16384 + 8192, &p.map_q, &bars->tma_full[st], cb * 64, h, tok, (int)b);
                tma_load_4d(dst + OFF_V + cb * 8192, &p.map_v, &bars->tma_full[st], cb * 64, h, tok, (int)b);
            }
            issued = c + 1;
        }
        // the last loads have landed before the CTA can leave (bounded; matters after an abort)
        for (int cc = max(0, issued - NSTAGE); cc < issued; ++cc) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_sleep(&bars->tma_full[cc % NSTAGE], (cc / NSTAGE) & 1, 20000) &&
                   globaltimer_ns() - t0 < WAIT_NS) {
            }
        }
    } else if (warp == 8) {
        // =============================== MMA warp ===============================
        // The whole warp runs this role converged; one elected lane issues each tcgen05
        // instruction (faster than a lone thread in a divergent branch).  Its issue loops are
        // fully unrolled, so the descriptors fold to constants.
        bool ok = true;
        // Gram products of full chunks up to `limit`, each once the prep has read the
        // previous one (one TM_G buffer) and the chunk's tile has landed.  With `block`
        // false it issues only what is ready now and never waits.
        int g_next = 0;
        auto issue_grams = [&](int limit, bool block) {
            while (ok && g_next <= limit && g_next < nchunks && eos - (bos + (long)g_next * C) >= C) {
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
                {
                    const uint32_t kq = s_sm + OFF_STAGE + (g_next % NSTAGE) * STAGE_BYTES;
                    const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16_e(tmem + TM_G, smem_desc(kq + off, 16, 1024), smem_desc(kq + off, 16, 1024), idesc,
                                   ks > 0);
                    }
                    mma_commit_e(&bars->g_done);
                }
                ++g_next;
            }
        };
        if (p.debug_stall) ok = wait_bar_warp(&bars->never, 0, abort_flag, wait_ns);
        issue_grams(0, true);
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c % NSTAGE, buf = c & 1;
            const uint32_t kq_s = s_sm + OFF_STAGE + st * STAGE_BYTES;
            const uint32_t tp = s_sm + OFF_TPP + buf * TPP_BYTES, pb = tp + 16384;
            // X needs the stage and the state only; a partial chunk also needs its zeroed tail,
            // which its prep writes before prep_ready
            const bool partial = eos - (bos + (long)c * C) < C;
            if (!(ok = wait_bar_warp(partial ? &bars->prep_ready[buf] : &bars->tma_full[st],
                                     partial ? (c >> 1) & 1 : (c / NSTAGE) & 1, abort_flag, wait_ns)))
                break;
            if (!(ok = wait_bar_warp(&bars->sa_ready, c & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            const uint32_t idesc64 = idesc_bf16_f32(128, 64, 0, 0);
            {  // X^T = S^T K^T (the chain): issued as soon as the S^T operand is written
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_bf16_ts_e(tmem + TM_X, tmem + TM_SA + part * 64 + ks * 8, smem_desc(kq_s + off, 16, 1024),
                                      idesc64, (part | ks) != 0);
                    }
                mma_commit_e(&bars->x_done);
            }
            issue_grams(c + 1, false);  // the next chunk's Gram product, if its inputs are ready
            // O1^T = S^T Q^T (off the chain) into this chunk's O^T buffer, once chunk c - 2's
            // outputs have been read out of it
            const uint32_t ob = TM_O + (uint32_t)(c & 1) * 64;
            if (write_o) {
                if (c >= 2 && !(ok = wait_bar_warp(&bars->o_free[c & 1], ((c - 2) >> 1) & 1, abort_flag, wait_ns)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32 + 8192;
                        mma_bf16_ts_e(tmem + ob, tmem + TM_SA + part * 64 + ks * 8, smem_desc(kq_s + off, 16, 1024),
                                      idesc64, (part | ks) != 0);
                    }
            }
            // the rest of the chunk needs its prep (T'', P)
            if (!(ok = wait_bar_warp(&bars->prep_ready[buf], (c >> 1) & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            issue_grams(c + 1, true);
            if (!ok) break;
            {  // [U1 | U2] = V^T [T''_hi; T''_lo]^T while the state warpgroup forms -X.  It
               // overwrites the S^T operand columns, which the products above (issued
               // earlier, executed in order) have already read.
                const uint32_t idesc = idesc_bf16_f32(128, 128, 1, 0);
                const uint32_t v_s = kq_s + OFF_V;
                if (mode != 1) {  // (the map from S = I takes v = 0)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_e(tmem + TM_SA, smem_desc(v_s + ks * 2048, 8192, 1024),
                                   smem_desc(tp + ks * 32, 16, 1024), idesc, ks > 0);
                }
            }
            if (!(ok = wait_bar_warp(&bars->r_ready, c & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            {  // u^T = [U1 | U2] + (-X)_hi^T [T''_hi; T''_lo]^T + (-X)_lo^T T''_hi^T  (u = U1 + U2)
                const uint32_t idesc2 = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts_e(tmem + TM_SA, tmem + TM_X + ks * 8, smem_desc(tp + ks * 32, 16, 1024), idesc2,
                                  mode != 1 || ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts_e(tmem + TM_SA, tmem + TM_X + 32 + ks * 8, smem_desc(tp + ks * 32, 16, 1024), idesc64,
                                  1);
                mma_commit_e(&bars->u_done);
            }
            // the Gram products two chunks ahead execute while the state warpgroup forms u
            issue_grams(c + 2, false);
            if (!(ok = wait_bar_warp(&bars->u_ready, c & 1, abort_flag, wait_ns))) break;
            tc_fence_after();
            {  // S^T += u^T K  (the chain), then O^T += u^T P^T
                const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_e(tmem + TM_S, tmem + TM_X + part * 32 + ks * 8,
                                      smem_desc(kq_s + ks * 2048, 16384, 1024), idesc_s, 1);
                mma_commit_e(&bars->s_done);
                mma_commit_e(&bars->s_free[c % NSTAGE]);
                // O^T += u_hi^T P_hi^T + u_hi^T P_lo^T + u_lo^T P_hi^T (N = 64 each)
                if (write_o) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_e(tmem + ob, tmem + TM_X + ks * 8, smem_desc(pb + ks * 32, 16, 1024), idesc64, 1);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_e(tmem + ob, tmem + TM_X + ks * 8, smem_desc(pb + 8192 + ks * 32, 16, 1024),
                                      idesc64, 1);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts_e(tmem + ob, tmem + TM_X + 32 + ks * 8, smem_desc(pb + ks * 32, 16, 1024),
                                      idesc64, 1);
                }
                mma_commit_e(&bars->o_done[c & 1]);
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

// 4-D map over a [B, T, H, 128] tensor: box of `box_x` features x 1 head x 64 tokens.
bool make_map(CUtensorMap *m, const void *ptr, int B, int T, int H, bool f32, int box_x, bool swizzle,
              int box_t = C) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es_b = f32 ? 4 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * es_b, (cuuint64_t)H * D * es_b, (cuuint64_t)T * H * D * es_b};
    cuuint32_t box[4] = {(cuuint32_t)box_x, 1, (cuuint32_t)box_t, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool OUT_BF16>
cudaError_t launch_typed(const TcParams &p, unsigned grid, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(chunk_tc_kernel<OUT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_done[dev] = true;
    }
    chunk_tc_kernel<OUT_BF16><<<grid, 448, SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_tc(const FwdArgs &a, const char **why) {
    if (a.N == 0) return cudaSuccess;
    TcParams p;
    memset(&p, 0, sizeof p);
    const bool o_bf16 = a.o_dtype == EFLA_BF16;
    if ((long long)a.B * a.T > 0) {
        if (!make_map(&p.map_q, a.q, a.B, a.T, a.H, false, 64, true) ||
            !make_map(&p.map_k, a.k, a.B, a.T, a.H, false, 64, true) ||
            !make_map(&p.map_v, a.v, a.B, a.T, a.H, false, 64, true) ||
            (a.o && !make_map(&p.map_o, a.o, a.B, a.T, a.H, !o_bf16, 32, false, o_bf16 ? 64 : 32))) {
            *why = "cuTensorMapEncodeTiled failed";
            return cudaErrorInvalidValue;
        }
    }
    p.beta = a.beta;
    p.S0 = a.S0;
    p.cu_seqlens = a.cu_seqlens;
    p.o = a.o;
    p.S_T = a.S_T;
    p.status = a.status;
    p.B = a.B;
    p.T = a.T;
    p.H = a.H;
    p.N = a.N;
    p.euler = a.euler;
    p.seg_len = a.seg_len;
    p.G = a.G;
    p.s_in = a.s_in;
    p.maps = a.maps;
    p.states = a.states;
    p.tpp = a.tpp;
    p.wait_ns = wait_limit_ns();
    p.debug_stall = (debug_stall() & STALL_CHUNK) ? 1 : 0;
    *why = "tcgen05 chunk kernel launch";
    const long units = a.seg_len > 0 ? (a.maps ? 2L * a.B * (a.G - 1) * a.H : (long)a.B * a.G * a.H) : (long)a.N * a.H;
    const unsigned grid = (unsigned)units;
    return o_bf16 ? launch_typed<true>(p, grid, a.stream) : launch_typed<false>(p, grid, a.stream);
}

}  // namespace efla
