// Chunked backward of the EFLA forward (chunks of C = 64 tokens), fp32 on CUDA cores.
//
// The pages give no backward formulas.  This is reverse mode of the chunkwise form of the
// recurrence ["Exact Flow Linear Attention" (gist.science), Metodologia 3; "Error-Free Linear
// Attention is a Free Lunch" (howistudyai), Steps 1-4]: for a chunk with start state S, keys K,
// queries Q, values V (C x d), alpha_t = f(beta_t, lambda_t), lambda_t = ||k_t||^2,
//   Ab = K K^T,  L = strictly-lower(Ab),  T = (I + diag(alpha) L)^{-1},  W = T diag(alpha)
//   R = V - K S,  U = W R,  P = (Q K^T) o M_incl,  O = Q S + P U,  S' = S + K^T U.
// Given dO and dS' (the gradient of the loss with respect to the chunk's end state):
//   G   = P^T dO + K dS'                     dR = W^T G       (dV = dR)
//   dY  = G - L^T dR                         Z  = R - L U
//   dalpha_t = sum_j dY[t][j] Z[t][j]
//   dP  = (dO U^T) o M_incl                  dL = -strictly-lower(dR U^T)
//   dQ  = dO S^T + dP K
//   dK  = -dR S^T + U dS'^T + dP^T Q + (dL + dL^T) K + 2 (dalpha o dalpha/dlambda) K
//   dbeta_t = dalpha_t dalpha/dbeta
//   dS  = dS' + Q^T dO - K^T dR               (the gradient with respect to the start state S)
// (dY = T^T G is written through dR = diag(alpha) dY, so no division by alpha is needed.)
//
// Three launches: the forward with the chunk-start states written out (the chunk kernels'
// `states` output), then
//   bwd_state_kernel: one CTA per (b, h) walks the chunks in reverse and writes dS' of every
//     chunk (the only serial part: dS' -> G -> dR -> dS);
//   bwd_grad_kernel:  one CTA per (b, h, chunk), all independent, forms every gradient above
//     from the chunk's S and dS'.
// W is formed with the normalized keys of the forward kernels (T'' = diag(1/n) T~ diag(gamma/n),
// T~ = (I + A~)^{-1}, A~ = strictly-lower(gamma_t k^_t . k^_s)), the same matrix as T diag(alpha).
#include "internal.cuh"
#include "tri_inverse.cuh"

namespace efla {
namespace {

constexpr int C = 64;
constexpr int NT = 256;
constexpr int LC = C + 4;  // row stride of the C x C matrices (a multiple of 4 for the inverse)
constexpr int J = 32;      // d_v columns per slab in bwd_grad_kernel
constexpr int LJ = J + 4;  // row stride of the slab matrices

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// A ROWS x COLS block of a row-major tensor (row stride `stride` elements) in 16-byte vectors,
// rows at or past `valid` as zeros: fetch() issues every load of the calling thread into
// registers, put() converts to fp32 and stores into shared memory [ROWS][ld].  Several
// fetches before their puts keep all of those loads in flight at once.
template <typename TIn, int ROWS, int COLS>
struct Block {
    static constexpr int VE = 16 / sizeof(TIn);  // elements per vector
    static constexpr int VPR = COLS / VE;        // vectors per row
    static constexpr int NV = ROWS * VPR / NT;   // vectors per thread
    static_assert(ROWS * VPR % NT == 0, "block must split evenly over the threads");
    uint4 r[NV];
    __device__ __forceinline__ void fetch(const TIn *src, size_t stride, int valid) {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            const int v = threadIdx.x + n * NT, row = v / VPR, col = (v % VPR) * VE;
            r[n] = row < valid ? __ldg(reinterpret_cast<const uint4 *>(src + (size_t)row * stride + col))
                               : make_uint4(0, 0, 0, 0);
        }
    }
    __device__ __forceinline__ void put(float *dst, int ld) const {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            const int v = threadIdx.x + n * NT, row = v / VPR, col = (v % VPR) * VE;
            float *d = dst + row * ld + col;
            if constexpr (sizeof(TIn) == 4) {
                st4(d, make_float4(__uint_as_float(r[n].x), __uint_as_float(r[n].y), __uint_as_float(r[n].z),
                                   __uint_as_float(r[n].w)));
            } else {
                const uint32_t w[4] = {r[n].x, r[n].y, r[n].z, r[n].w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = __uint_as_float(w[e] << 16);
                    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                }
                st4(d, make_float4(f[0], f[1], f[2], f[3]));
                st4(d + 4, make_float4(f[4], f[5], f[6], f[7]));
            }
        }
    }
};

// Ab[t][s] = k_t . k_s and Pm[t][s] = q_t . k_s for s <= t (0 above), [C][LD]; thread tile
// rows r4 + 16 r, columns c4 + 16 c (r, c < 4).
template <int D, int LD>
__device__ __forceinline__ void gram(const float *Ks, const float *Qs, int ldk, float *Ab, float *Pm) {
    const int r4 = threadIdx.x >> 4, c4 = threadIdx.x & 15;
    float kk[4][4] = {}, qk[4][4] = {};
#pragma unroll 2
    for (int i = 0; i < D; i += 4) {
        float4 kt[4], qt[4], ks[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            kt[r] = ld4(Ks + (r4 + 16 * r) * ldk + i);
            qt[r] = ld4(Qs + (r4 + 16 * r) * ldk + i);
            ks[r] = ld4(Ks + (c4 + 16 * r) * ldk + i);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                kk[r][c] = fmaf(kt[r].x, ks[c].x, fmaf(kt[r].y, ks[c].y, fmaf(kt[r].z, ks[c].z, fmaf(kt[r].w, ks[c].w, kk[r][c]))));
                qk[r][c] = fmaf(qt[r].x, ks[c].x, fmaf(qt[r].y, ks[c].y, fmaf(qt[r].z, ks[c].z, fmaf(qt[r].w, ks[c].w, qk[r][c]))));
            }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int t = r4 + 16 * r, s = c4 + 16 * c;
            Ab[t * LD + s] = kk[r][c];
            Pm[t * LD + s] = s <= t ? qk[r][c] : 0.f;
        }
}

// ============================ state gradients (serial over chunks) ============================
// Shared memory (floats): K [C][D+4]; Q, dO [C][D]; G, then dR in place [C][D]; Pm [C][C];
// W [C][LC] (A~, then T~ in place, then W); per-row gate terms 3 x [C]; dS [D][D]
// (226.75 KB at D = 128).
constexpr int LCS = C;  // row stride of Pm here (read along columns only)
template <int D>
constexpr size_t state_smem_floats() {
    return (size_t)C * (D + 4) + 3 * (size_t)C * D + (size_t)C * LCS + (size_t)C * LC + 3 * C + (size_t)D * D;
}

// W = diag(1/n) T~ diag(gamma/n) in place over T~ (lower triangle; zero above), with a zero
// key's row keeping u_t = alpha_t r_t (W[t][t] = alpha_t).
__device__ __forceinline__ void form_w(float *W, const float *invn, const float *gn, const float *al) {
    for (int e = threadIdx.x; e < C * C; e += NT) {
        const int t = e / C, s = e % C;
        const float w = s < t ? invn[t] * W[t * LC + s] * gn[s] : s == t ? (invn[t] > 0.f ? gn[t] * invn[t] : al[t]) : 0.f;
        W[t * LC + s] = w;  // (each thread reads only the element it writes)
    }
}

template <typename TIn, int D>
__global__ void __launch_bounds__(NT, 1) bwd_state_kernel(BwdArgs a, float *dse) {
    extern __shared__ __align__(16) float sm[];
    constexpr int LK = D + 4;
    constexpr int TN = D / 16;  // columns of G / dR per thread
    float *Ks = sm, *Qs = Ks + C * LK, *dOs = Qs + C * D, *Gs = dOs + C * D, *Pm = Gs + C * D, *W = Pm + C * LCS;
    float *al = W + C * LC, *invn = al + C, *gn = invn + C, *dS = gn + C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int nc = (a.T + C - 1) / C;
    const size_t ubase = (size_t)blockIdx.x * D * D;
    const TIn *q = static_cast<const TIn *>(a.q);
    const TIn *k = static_cast<const TIn *>(a.k);
    for (int e = tid; e < D * D; e += NT) dS[e] = a.dST ? a.dST[ubase + e] : 0.f;
    // G / dR tile: rows r4 + 16 r, columns TN c16 .. TN c16 + TN - 1
    const int r4 = tid >> 4, c16 = tid & 15;

    for (int c = nc - 1; c >= 0; --c) {
        const long t0 = (long)c * C;
        const int valid = (int)min((long)C, (long)a.T - t0);
        __syncthreads();  // the previous chunk is done with every buffer; dS is complete
        {  // the gradient with respect to this chunk's end state
            float *dst = dse + ((size_t)blockIdx.x * nc + c) * D * D;
            for (int e = 4 * tid; e < D * D; e += 4 * NT) st4(dst + e, ld4(dS + e));
        }
        {
            const size_t row0 = ((size_t)b * a.T + (size_t)t0) * a.H + h, stride = (size_t)a.H * D;
            Block<TIn, C, D> kb, qb;
            Block<float, C, D> ob;
            kb.fetch(k + row0 * D, stride, valid);
            qb.fetch(q + row0 * D, stride, valid);
            ob.fetch(a.dO + row0 * D, stride, valid);
            kb.put(Ks, LK);
            qb.put(Qs, D);
            ob.put(dOs, D);
        }
        __syncthreads();
        for (int t = warp; t < C; t += NT / 32) {  // gate terms from lambda_t = ||k_t||^2
            float lam = 0.f;
            for (int i = lane; i < D; i += 32) lam = fmaf(Ks[t * LK + i], Ks[t * LK + i], lam);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
            if (lane == 0) {
                const float bt = t < valid ? a.beta[((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h] : 0.f;
                const bool live = t < valid && lam > 0.f;
                const float in = live ? rsqrtf(lam) : 0.f;
                const float gam = !live ? 0.f : a.euler ? bt * lam : -expm1f(-bt * lam);
                al[t] = t < valid ? efla_alpha(bt, lam, a.euler) : 0.f;
                invn[t] = in;
                gn[t] = gam * in;
            }
        }
        __syncthreads();
        {  // A~ = strictly-lower(gamma_t/n_t (k_t . k_s) / n_s) into W and P = (Q K^T) o M_incl into Pm
            float kk[4][4] = {}, qk[4][4] = {};
#pragma unroll 2
            for (int i = 0; i < D; i += 4) {
                float4 kt[4], qt[4], ks[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    kt[r] = ld4(Ks + (r4 + 16 * r) * LK + i);
                    qt[r] = ld4(Qs + (r4 + 16 * r) * D + i);
                    ks[r] = ld4(Ks + (c16 + 16 * r) * LK + i);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        kk[r][cc] = fmaf(kt[r].x, ks[cc].x, fmaf(kt[r].y, ks[cc].y, fmaf(kt[r].z, ks[cc].z, fmaf(kt[r].w, ks[cc].w, kk[r][cc]))));
                        qk[r][cc] = fmaf(qt[r].x, ks[cc].x, fmaf(qt[r].y, ks[cc].y, fmaf(qt[r].z, ks[cc].z, fmaf(qt[r].w, ks[cc].w, qk[r][cc]))));
                    }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int t = r4 + 16 * r, s = c16 + 16 * cc;
                    W[t * LC + s] = s < t ? gn[t] * kk[r][cc] * invn[s] : 0.f;
                    Pm[t * LCS + s] = s <= t ? qk[r][cc] : 0.f;
                }
        }
        __syncthreads();
        invert_unit_lower<1, LC>(W, tid);  // ends with a barrier over all 256 threads
        form_w(W, invn, gn, al);
        float acc[4][TN] = {};
        {  // G[t][j] = sum_i K[t][i] dS[i][j] + sum_{s >= t} P[s][t] dO[s][j]
#pragma unroll 1
            for (int i = 0; i < D; i += 4) {
                float4 kt[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) kt[r] = ld4(Ks + (r4 + 16 * r) * LK + i);
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    float sv[TN];
#pragma unroll
                    for (int n = 0; n < TN; n += 4) *reinterpret_cast<float4 *>(sv + n) = ld4(dS + (i + ii) * D + TN * c16 + n);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float kv = ii == 0 ? kt[r].x : ii == 1 ? kt[r].y : ii == 2 ? kt[r].z : kt[r].w;
#pragma unroll
                        for (int n = 0; n < TN; ++n) acc[r][n] = fmaf(kv, sv[n], acc[r][n]);
                    }
                }
            }
#pragma unroll 1
            for (int s = 0; s < valid; ++s) {
                float ov[TN];
#pragma unroll
                for (int n = 0; n < TN; n += 4) *reinterpret_cast<float4 *>(ov + n) = ld4(dOs + s * D + TN * c16 + n);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float pv = Pm[s * LCS + r4 + 16 * r];  // P[s][t], zero for t > s
#pragma unroll
                    for (int n = 0; n < TN; ++n) acc[r][n] = fmaf(pv, ov[n], acc[r][n]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int n = 0; n < TN; n += 4)
                    st4(Gs + (r4 + 16 * r) * D + TN * c16 + n, make_float4(acc[r][n], acc[r][n + 1], acc[r][n + 2], acc[r][n + 3]));
        }
        __syncthreads();  // G and W complete
        {  // dR = W^T G: dR[t][j] = sum_{s >= t} W[s][t] G[s][j], written over G once all of G is read
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int n = 0; n < TN; ++n) acc[r][n] = 0.f;
#pragma unroll 1
            for (int s = 0; s < valid; ++s) {
                float gv[TN];
#pragma unroll
                for (int n = 0; n < TN; n += 4) *reinterpret_cast<float4 *>(gv + n) = ld4(Gs + s * D + TN * c16 + n);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float wv = W[s * LC + r4 + 16 * r];  // W[s][t], zero for s < t
#pragma unroll
                    for (int n = 0; n < TN; ++n) acc[r][n] = fmaf(wv, gv[n], acc[r][n]);
                }
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int n = 0; n < TN; n += 4)
                    st4(Gs + (r4 + 16 * r) * D + TN * c16 + n, make_float4(acc[r][n], acc[r][n + 1], acc[r][n + 2], acc[r][n + 3]));
        }
        __syncthreads();
        {  // dS += Q^T dO - K^T dR; rows TI i16 .., columns TI j16 ..
            constexpr int TI = D / 16;
            const int i16 = tid >> 4, j16 = tid & 15;
            float sacc[TI][TI];
#pragma unroll
            for (int r = 0; r < TI; ++r)
#pragma unroll
                for (int n = 0; n < TI; n += 4) {
                    const float4 v = ld4(dS + (TI * i16 + r) * D + TI * j16 + n);
                    sacc[r][n] = v.x;
                    sacc[r][n + 1] = v.y;
                    sacc[r][n + 2] = v.z;
                    sacc[r][n + 3] = v.w;
                }
#pragma unroll 1
            for (int t = 0; t < valid; ++t) {
                float qv[TI], kv[TI], ov[TI], rv[TI];
#pragma unroll
                for (int n = 0; n < TI; n += 4) {
                    *reinterpret_cast<float4 *>(qv + n) = ld4(Qs + t * D + TI * i16 + n);
                    *reinterpret_cast<float4 *>(kv + n) = ld4(Ks + t * LK + TI * i16 + n);
                    *reinterpret_cast<float4 *>(ov + n) = ld4(dOs + t * D + TI * j16 + n);
                    *reinterpret_cast<float4 *>(rv + n) = ld4(Gs + t * D + TI * j16 + n);
                }
#pragma unroll
                for (int r = 0; r < TI; ++r)
#pragma unroll
                    for (int n = 0; n < TI; ++n) sacc[r][n] = fmaf(qv[r], ov[n], fmaf(-kv[r], rv[n], sacc[r][n]));
            }
#pragma unroll
            for (int r = 0; r < TI; ++r)
#pragma unroll
                for (int n = 0; n < TI; n += 4)
                    st4(dS + (TI * i16 + r) * D + TI * j16 + n, make_float4(sacc[r][n], sacc[r][n + 1], sacc[r][n + 2], sacc[r][n + 3]));
        }
    }
    __syncthreads();
    if (a.dS0)
        for (int e = 4 * tid; e < D * D; e += 4 * NT) st4(a.dS0 + ubase + e, ld4(dS + e));
}

// ============================ per-chunk gradients (parallel) ============================
// Shared memory (floats): K, Q [C][D+4]; Ab, Pm, W [C][LC]; per-row gate terms 6 x [C];
// slabs S, dS' [D][LJ] and V, dO, R, U, G, dR [C][LJ].
template <int D>
constexpr size_t grad_smem_floats() {
    return 2 * (size_t)C * (D + 4) + 3 * (size_t)C * LC + 6 * C + 2 * (size_t)D * LJ + 6 * (size_t)C * LJ;
}

template <typename TIn, int D>
__global__ void __launch_bounds__(NT, 1) bwd_grad_kernel(BwdArgs a, const float *states, const float *dse) {
    extern __shared__ __align__(16) float sm[];
    constexpr int LK = D + 4;
    constexpr int TI = D / 16;  // columns of dQ / dK per thread
    float *Ks = sm, *Qs = Ks + C * LK, *Ab = Qs + C * LK, *Pm = Ab + C * LC, *W = Pm + C * LC;
    float *al = W + C * LC, *invn = al + C, *gn = invn + C, *dadb = gn + C, *dadl = dadb + C, *dal = dadl + C;
    float *Ssl = dal + C, *dSsl = Ssl + D * LJ, *Vsl = dSsl + D * LJ, *dOsl = Vsl + C * LJ, *Rs = dOsl + C * LJ;
    float *Us = Rs + C * LJ, *Gs = Us + C * LJ, *dRs = Gs + C * LJ;
    const int tid = threadIdx.x;
    const int nc = (a.T + C - 1) / C;
    const int unit = blockIdx.x / nc, c = blockIdx.x % nc;
    const int b = unit / a.H, h = unit % a.H;
    const long t0 = (long)c * C;
    const int valid = (int)min((long)C, (long)a.T - t0);
    const float *Sc = states + (size_t)blockIdx.x * D * D;
    const float *dSe = dse + (size_t)blockIdx.x * D * D;
    const TIn *q = static_cast<const TIn *>(a.q);
    const TIn *k = static_cast<const TIn *>(a.k);
    const TIn *v = static_cast<const TIn *>(a.v);

    const size_t row0 = ((size_t)b * a.T + (size_t)t0) * a.H + h, stride = (size_t)a.H * D;
    {
        Block<TIn, C, D> kb, qb;
        kb.fetch(k + row0 * D, stride, valid);
        qb.fetch(q + row0 * D, stride, valid);
        kb.put(Ks, LK);
        qb.put(Qs, LK);
    }
    __syncthreads();
    gram<D, LC>(Ks, Qs, LK, Ab, Pm);
    __syncthreads();
    if (tid < C) {  // gate terms of row t
        const int t = tid;
        const float lam = Ab[t * LC + t];
        const float bt = t < valid ? a.beta[((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h] : 0.f;
        const bool live = t < valid && lam > 0.f;
        const float in = live ? rsqrtf(lam) : 0.f;
        const float gam = !live ? 0.f : a.euler ? bt * lam : -expm1f(-bt * lam);
        float db = 0.f, dl = 0.f;
        if (t < valid) gate_grad(bt, lam, a.euler, db, dl);
        al[t] = t < valid ? efla_alpha(bt, lam, a.euler) : 0.f;
        invn[t] = in;
        gn[t] = gam * in;
        dadb[t] = db;
        dadl[t] = dl;
        dal[t] = 0.f;
    }
    __syncthreads();
    for (int e = tid; e < C * C; e += NT) {  // A~ = strictly-lower(gamma_t k^_t . k^_s) into W
        const int t = e / C, s = e % C;
        W[t * LC + s] = s < t ? gn[t] * Ab[t * LC + s] * invn[s] : 0.f;
    }
    __syncthreads();
    invert_unit_lower<1, LC>(W, tid);  // ends with a barrier over all 256 threads
    form_w(W, invn, gn, al);
    __syncthreads();

    // slab thread tile: row ts = tid / 4, columns jq .. jq + 7
    const int ts = tid >> 2, jq = (tid & 3) * 8;
    // accumulator tiles: dP, dLr [C][C] rows r4 + 16 r, cols c4 + 16 cc; dQ, dK [C][D] rows r4 + 16 r, cols c4 + 16 cc
    const int r4 = tid >> 4, c4 = tid & 15;
    float dP[4][4] = {}, dLr[4][4] = {}, dQ[4][TI] = {}, dK[4][TI] = {};
    float dal_part = 0.f;

#pragma unroll 1
    for (int j0 = 0; j0 < D; j0 += J) {
        __syncthreads();  // the previous slab's buffers are free
        {
            Block<float, D, J> sb, eb;
            Block<TIn, C, J> vb;
            Block<float, C, J> ob;
            sb.fetch(Sc + j0, D, D);
            eb.fetch(dSe + j0, D, D);
            vb.fetch(v + row0 * D + j0, stride, valid);
            ob.fetch(a.dO + row0 * D + j0, stride, valid);
            sb.put(Ssl, LJ);
            eb.put(dSsl, LJ);
            vb.put(Vsl, LJ);
            ob.put(dOsl, LJ);
        }
        __syncthreads();
        {  // R = V - K S and G = P^T dO + K dS' (row ts, columns jq ..)
            float x[8] = {}, g[8] = {};
#pragma unroll 1
            for (int i = 0; i < D; i += 4) {
                const float4 kt = ld4(Ks + ts * LK + i);
                const float kv[4] = {kt.x, kt.y, kt.z, kt.w};
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const float4 s0 = ld4(Ssl + (i + ii) * LJ + jq), s1 = ld4(Ssl + (i + ii) * LJ + jq + 4);
                    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                    for (int n = 0; n < 8; ++n) x[n] = fmaf(kv[ii], sv[n], x[n]);
                    const float4 d0 = ld4(dSsl + (i + ii) * LJ + jq), d1 = ld4(dSsl + (i + ii) * LJ + jq + 4);
                    const float dv8[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                    for (int n = 0; n < 8; ++n) g[n] = fmaf(kv[ii], dv8[n], g[n]);
                }
            }
#pragma unroll 1
            for (int s = ts; s < valid; ++s) {  // P[s][ts] is zero for s < ts
                const float pv = Pm[s * LC + ts];
                const float4 o0 = ld4(dOsl + s * LJ + jq), o1 = ld4(dOsl + s * LJ + jq + 4);
                const float ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
                for (int n = 0; n < 8; ++n) g[n] = fmaf(pv, ov[n], g[n]);
            }
            const float4 v0 = ld4(Vsl + ts * LJ + jq), v1 = ld4(Vsl + ts * LJ + jq + 4);
            st4(Rs + ts * LJ + jq, make_float4(v0.x - x[0], v0.y - x[1], v0.z - x[2], v0.w - x[3]));
            st4(Rs + ts * LJ + jq + 4, make_float4(v1.x - x[4], v1.y - x[5], v1.z - x[6], v1.w - x[7]));
            st4(Gs + ts * LJ + jq, make_float4(g[0], g[1], g[2], g[3]));
            st4(Gs + ts * LJ + jq + 4, make_float4(g[4], g[5], g[6], g[7]));
        }
        __syncthreads();
        {  // U = W R (W lower) and dR = W^T G (W^T upper)
            float u[8] = {}, r[8] = {};
#pragma unroll 1
            for (int s = 0; s <= ts; ++s) {
                const float wv = W[ts * LC + s];
                const float4 a0 = ld4(Rs + s * LJ + jq), a1 = ld4(Rs + s * LJ + jq + 4);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int n = 0; n < 8; ++n) u[n] = fmaf(wv, av[n], u[n]);
            }
#pragma unroll 1
            for (int s = ts; s < C; ++s) {
                const float wv = W[s * LC + ts];
                const float4 a0 = ld4(Gs + s * LJ + jq), a1 = ld4(Gs + s * LJ + jq + 4);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int n = 0; n < 8; ++n) r[n] = fmaf(wv, av[n], r[n]);
            }
            st4(Us + ts * LJ + jq, make_float4(u[0], u[1], u[2], u[3]));
            st4(Us + ts * LJ + jq + 4, make_float4(u[4], u[5], u[6], u[7]));
            st4(dRs + ts * LJ + jq, make_float4(r[0], r[1], r[2], r[3]));
            st4(dRs + ts * LJ + jq + 4, make_float4(r[4], r[5], r[6], r[7]));
            if (ts < valid) {  // dv = dR
                float *dvp = a.dv + (((size_t)b * a.T + (size_t)(t0 + ts)) * a.H + h) * D + j0 + jq;
                st4(dvp, make_float4(r[0], r[1], r[2], r[3]));
                st4(dvp + 4, make_float4(r[4], r[5], r[6], r[7]));
            }
        }
        __syncthreads();
        {  // dalpha_t += sum_j (G - L^T dR)[t][j] (R - L U)[t][j]
            float y[8], z[8];
            {
                const float4 g0 = ld4(Gs + ts * LJ + jq), g1 = ld4(Gs + ts * LJ + jq + 4);
                const float4 q0 = ld4(Rs + ts * LJ + jq), q1 = ld4(Rs + ts * LJ + jq + 4);
                const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                const float rv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    y[n] = gv[n];
                    z[n] = rv[n];
                }
            }
#pragma unroll 1
            for (int s = ts + 1; s < valid; ++s) {
                const float lv = Ab[s * LC + ts];
                const float4 a0 = ld4(dRs + s * LJ + jq), a1 = ld4(dRs + s * LJ + jq + 4);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int n = 0; n < 8; ++n) y[n] = fmaf(-lv, av[n], y[n]);
            }
#pragma unroll 1
            for (int s = 0; s < ts; ++s) {
                const float lv = Ab[ts * LC + s];
                const float4 a0 = ld4(Us + s * LJ + jq), a1 = ld4(Us + s * LJ + jq + 4);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int n = 0; n < 8; ++n) z[n] = fmaf(-lv, av[n], z[n]);
            }
            float acc = 0.f;
#pragma unroll
            for (int n = 0; n < 8; ++n) acc = fmaf(y[n], z[n], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            dal_part += acc;  // the same in the 4 threads of row ts
        }
        {  // dP += dO U^T, dLr += dR U^T (over this slab's columns)
#pragma unroll 1
            for (int jj = 0; jj < J; jj += 4) {
                float4 o4[4], r4v[4], u4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    o4[r] = ld4(dOsl + (r4 + 16 * r) * LJ + jj);
                    r4v[r] = ld4(dRs + (r4 + 16 * r) * LJ + jj);
                    u4[r] = ld4(Us + (c4 + 16 * r) * LJ + jj);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        dP[r][cc] = fmaf(o4[r].x, u4[cc].x, fmaf(o4[r].y, u4[cc].y, fmaf(o4[r].z, u4[cc].z, fmaf(o4[r].w, u4[cc].w, dP[r][cc]))));
                        dLr[r][cc] = fmaf(r4v[r].x, u4[cc].x, fmaf(r4v[r].y, u4[cc].y, fmaf(r4v[r].z, u4[cc].z, fmaf(r4v[r].w, u4[cc].w, dLr[r][cc]))));
                    }
            }
        }
        {  // dQ += dO S^T, dK += -dR S^T + U dS'^T (over this slab's columns)
#pragma unroll 1
            for (int jj = 0; jj < J; jj += 4) {
                float4 o4[4], r4v[4], u4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    o4[r] = ld4(dOsl + (r4 + 16 * r) * LJ + jj);
                    r4v[r] = ld4(dRs + (r4 + 16 * r) * LJ + jj);
                    u4[r] = ld4(Us + (r4 + 16 * r) * LJ + jj);
                }
#pragma unroll
                for (int cc = 0; cc < TI; ++cc) {
                    const float4 s4 = ld4(Ssl + (c4 + 16 * cc) * LJ + jj);
                    const float4 e4 = ld4(dSsl + (c4 + 16 * cc) * LJ + jj);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        dQ[r][cc] = fmaf(o4[r].x, s4.x, fmaf(o4[r].y, s4.y, fmaf(o4[r].z, s4.z, fmaf(o4[r].w, s4.w, dQ[r][cc]))));
                        float x = dK[r][cc];
                        x = fmaf(-r4v[r].x, s4.x, fmaf(-r4v[r].y, s4.y, fmaf(-r4v[r].z, s4.z, fmaf(-r4v[r].w, s4.w, x))));
                        x = fmaf(u4[r].x, e4.x, fmaf(u4[r].y, e4.y, fmaf(u4[r].z, e4.z, fmaf(u4[r].w, e4.w, x))));
                        dK[r][cc] = x;
                    }
                }
            }
        }
    }
    __syncthreads();  // every slab done: Pm, Ab and W are free
    if ((tid & 3) == 0) dal[ts] = dal_part;
    // dP (inclusive lower) into Pm, dL = -strictly-lower(dLr) into W
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int t = r4 + 16 * r, s = c4 + 16 * cc;
            Pm[t * LC + s] = s <= t ? dP[r][cc] : 0.f;
            W[t * LC + s] = s < t ? -dLr[r][cc] : 0.f;
        }
    __syncthreads();
    for (int e = tid; e < C * C; e += NT) {  // dLsym = dL + dL^T into Ab
        const int t = e / C, s = e % C;
        Ab[t * LC + s] = W[t * LC + s] + W[s * LC + t];
    }
    __syncthreads();
    {  // dQ += dP K, dK += dP^T Q + dLsym K + 2 dalpha dalpha/dlambda k
#pragma unroll 1
        for (int s = 0; s < valid; ++s) {
            float pr[4], pc[4], lr[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = r4 + 16 * r;
                pr[r] = Pm[t * LC + s];  // dP[t][s]
                pc[r] = Pm[s * LC + t];  // dP[s][t]
                lr[r] = Ab[t * LC + s];  // dLsym[t][s]
            }
#pragma unroll
            for (int cc = 0; cc < TI; ++cc) {
                const float kv = Ks[s * LK + c4 + 16 * cc], qv = Qs[s * LK + c4 + 16 * cc];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    dQ[r][cc] = fmaf(pr[r], kv, dQ[r][cc]);
                    dK[r][cc] = fmaf(pc[r], qv, fmaf(lr[r], kv, dK[r][cc]));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = r4 + 16 * r;
            if (t >= valid) continue;
            const size_t row = ((size_t)b * a.T + (size_t)(t0 + t)) * a.H + h;
            const float dl2 = 2.f * dal[t] * dadl[t];
#pragma unroll
            for (int cc = 0; cc < TI; ++cc) {
                const int i = c4 + 16 * cc;
                a.dq[row * D + i] = dQ[r][cc];
                a.dk[row * D + i] = fmaf(dl2, Ks[t * LK + i], dK[r][cc]);
            }
        }
        if (tid < valid) a.dbeta[((size_t)b * a.T + (size_t)(t0 + tid)) * a.H + h] = dal[tid] * dadb[tid];
    }
}

static_assert(state_smem_floats<128>() * sizeof(float) <= 232448, "state kernel shared memory");
static_assert(grad_smem_floats<128>() * sizeof(float) <= 232448, "gradient kernel shared memory");

template <typename TIn, int D>
cudaError_t launch_d(const BwdArgs &a, const float *states, float *dse) {
    const int nc = (a.T + C - 1) / C;
    const size_t s1 = state_smem_floats<D>() * sizeof(float), s2 = grad_smem_floats<D>() * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(bwd_state_kernel<TIn, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_grad_kernel<TIn, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
    if (e != cudaSuccess) return e;
    bwd_state_kernel<TIn, D><<<(unsigned)((long)a.B * a.H), NT, s1, a.stream>>>(a, dse);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (nc == 0) return cudaSuccess;
    bwd_grad_kernel<TIn, D><<<(unsigned)((long)a.B * a.H * nc), NT, s2, a.stream>>>(a, states, dse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_chunked(const BwdArgs &a, const float *states, float *dse) {
    if ((long long)a.B * a.H == 0) return cudaSuccess;
    const bool bf = a.in_dtype == EFLA_BF16;
    if (a.dk_dim == 64)
        return bf ? launch_d<__nv_bfloat16, 64>(a, states, dse) : launch_d<float, 64>(a, states, dse);
    return bf ? launch_d<__nv_bfloat16, 128>(a, states, dse) : launch_d<float, 128>(a, states, dse);
}

}  // namespace efla
