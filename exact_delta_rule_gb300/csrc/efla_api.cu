// C-ABI entry points of libefla.so: argument validation, dispatch to the
// kernels, status reporting.  Declarations and the contract are in efla.h.
#include <stdarg.h>
#include <stdio.h>

#include <string>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.cuh"

namespace efla {
namespace {

__device__ int g_device_status = 0;

// Scratch of efla_fwd_chunked_scan_static: a fixed device array, so that call
// allocates nothing.  32 MiB holds the segment states and maps of any split the
// automatic segment count picks on a GPU of up to 170 SMs ((3 G - 2) B H pieces of
// 64 KiB with G <= SMs / (B H)).
constexpr size_t SCAN_SCRATCH_BYTES = 32ull << 20;
static __device__ __align__(256) unsigned char g_scan_scratch[SCAN_SCRATCH_BYTES];

thread_local std::string g_last_error;

efla_status fail(efla_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

efla_status cuda_fail(cudaError_t e, const char *what) {
    return fail(EFLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t dsize(efla_dtype t) { return t == EFLA_BF16 ? 2 : 4; }

struct Range {
    const char *name;
    uintptr_t lo, hi;
};
bool overlap(const Range &a, const Range &b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

efla_status check_dims_common(int d_k, int d_v, efla_dtype in_dtype, efla_dtype o_dtype) {
    if (d_k <= 0 || d_v <= 0) return fail(EFLA_ERR_INVALID_ARG, "d_k=%d d_v=%d must be positive", d_k, d_v);
    if (!supported_dim(d_k) || !supported_dim(d_v))
        return fail(EFLA_ERR_UNSUPPORTED, "d_k=%d d_v=%d: supported head sizes are 32, 64, 128", d_k, d_v);
    if ((in_dtype != EFLA_BF16 && in_dtype != EFLA_F32) || (o_dtype != EFLA_BF16 && o_dtype != EFLA_F32))
        return fail(EFLA_ERR_INVALID_ARG, "unknown dtype (in=%d, o=%d)", (int)in_dtype, (int)o_dtype);
    return EFLA_OK;
}

efla_status validate_fwd(const FwdArgs &a, bool chunked) {
    if (a.B < 0 || a.T < 0 || a.H <= 0 || a.N < 0)
        return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d N=%d", a.B, a.T, a.H, a.N);
    efla_status s = check_dims_common(a.dk, a.dv, a.in_dtype, a.o_dtype);
    if (s != EFLA_OK) return s;
    if (chunked && a.chunk != 16 && a.chunk != 32 && a.chunk != 64)
        return fail(EFLA_ERR_UNSUPPORTED, "chunk=%d: supported chunk lengths are 16, 32 and 64", a.chunk);
    if (a.cu_seqlens) {
        if (a.B != 1) return fail(EFLA_ERR_INVALID_ARG, "cu_seqlens given with B=%d (must be 1)", a.B);
    } else if (a.N != a.B) {
        return fail(EFLA_ERR_INVALID_ARG, "N=%d must equal B=%d when cu_seqlens is NULL", a.N, a.B);
    }
    const long long tokens = (long long)a.B * a.T;
    if (tokens * a.H > (1LL << 31) - 1)
        return fail(EFLA_ERR_UNSUPPORTED, "B*T*H=%lld exceeds 2^31-1 token-heads", tokens * a.H);
    if (a.cu_seqlens && a.N > (1 << 30)) return fail(EFLA_ERR_INVALID_ARG, "N=%d too large", a.N);
    if (tokens > 0 && (!a.q || !a.k || !a.v || !a.beta || !a.o))
        return fail(EFLA_ERR_INVALID_ARG, "q, k, v, beta and o must be non-NULL when B*T > 0");
    const void *ptrs[] = {a.q, a.k, a.v, a.beta, a.S0, a.cu_seqlens, a.o, a.S_T};
    const char *names[] = {"q", "k", "v", "beta", "S0", "cu_seqlens", "o", "S_T"};
    for (int i = 0; i < 8; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(EFLA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    const size_t th = (size_t)tokens * a.H;
    const size_t st = (size_t)a.N * a.H * a.dk * a.dv * 4;
    auto R = [](const char *n, const void *p, size_t bytes) {
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{n, lo, p ? lo + bytes : lo};
    };
    const Range in[] = {R("q", a.q, th * a.dk * dsize(a.in_dtype)), R("k", a.k, th * a.dk * dsize(a.in_dtype)),
                        R("v", a.v, th * a.dv * dsize(a.in_dtype)), R("beta", a.beta, th * 4),
                        R("S0", a.S0, st), R("cu_seqlens", a.cu_seqlens, a.cu_seqlens ? (size_t)(a.N + 1) * 4 : 0)};
    const Range out[] = {R("o", a.o, th * a.dv * dsize(a.o_dtype)), R("S_T", a.S_T, st)};
    for (const Range &w : out)
        for (const Range &r : in) {
            if (w.name[0] == 'S' && r.name[0] == 'S' && w.lo == r.lo) continue;  // S0 == S_T allowed
            if (overlap(w, r)) return fail(EFLA_ERR_INVALID_ARG, "output %s overlaps input %s", w.name, r.name);
        }
    if (overlap(out[0], out[1])) return fail(EFLA_ERR_INVALID_ARG, "o overlaps S_T");
    return EFLA_OK;
}

efla_status run_fwd(FwdArgs a, bool chunked) {
    efla_status s = validate_fwd(a, chunked);
    if (s != EFLA_OK) return s;
    a.status = device_status_ptr();
    if (!a.status) return fail(EFLA_ERR_CUDA, "cannot resolve the device status word");
    cudaError_t e;
    if (chunked && a.in_dtype == EFLA_BF16 && a.dk == 128 && a.dv == 128 && a.chunk == 64) {
        const char *why = nullptr;
        e = launch_chunk_tc(a, &why);
        if (e != cudaSuccess) return cuda_fail(e, why ? why : "tcgen05 chunk kernel launch");
    } else if (chunked) {
        e = launch_chunk_simt(a);
        if (e != cudaSuccess) return cuda_fail(e, "chunk kernel launch");
    } else {
        e = launch_recurrent(a);
        if (e != cudaSuccess) return cuda_fail(e, "recurrent kernel launch");
    }
    g_last_error.clear();
    return EFLA_OK;
}

}  // namespace

int *device_status_ptr() {
    // One status word per device: the symbol's device address differs per device, so it is
    // resolved (once) with that device current.
    static std::mutex mu;
    static int *ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        int *p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_device_status) == cudaSuccess) ptrs[dev] = p;
    }
    return ptrs[dev];
}

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{0};
std::atomic<int> g_debug_stall{0};
}

int debug_stall() { return g_debug_stall.load(std::memory_order_relaxed); }

unsigned long long wait_limit_ns() {
    const unsigned long long v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v ? v : 2000000000ull;
}

void set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }

}  // namespace efla

using namespace efla;

extern "C" {

static bool update_ok(efla_update u) { return u == EFLA_UPDATE_EXACT || u == EFLA_UPDATE_EULER; }

efla_status efla_fwd_chunked_ex(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                                const int32_t *cu_seqlens, void *o, float *S_T, int B, int T, int H, int d_k,
                                int d_v, int N, efla_dtype in_dtype, efla_dtype o_dtype, int chunk,
                                efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    FwdArgs a{q, k, v, beta, S0, cu_seqlens, o, S_T, B, T, H, d_k, d_v, N, in_dtype, o_dtype,
              chunk == 0 ? 64 : chunk, reinterpret_cast<cudaStream_t>(stream), nullptr, (int)update};
    return run_fwd(a, true);
}

efla_status efla_fwd_chunked(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                             const int32_t *cu_seqlens, void *o, float *S_T, int B, int T, int H, int d_k,
                             int d_v, int N, efla_dtype dtype, int chunk, efla_stream_t stream) {
    return efla_fwd_chunked_ex(q, k, v, beta, S0, cu_seqlens, o, S_T, B, T, H, d_k, d_v, N, dtype, dtype, chunk,
                               EFLA_UPDATE_EXACT, stream);
}

// Segments of the split forward: G segments of seg_len tokens (a multiple of the chunk)
// per sequence, every one non-empty.  segments <= 0 picks G = SMs / (B*H).
static efla_status scan_plan(int B, int T, int H, int segments, int *G_out, int *seg_len) {
    const int nch = (T + 63) / 64;
    int G = segments;
    if (G <= 0) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "querying the SM count");
        G = sms / (B * H > 0 ? B * H : 1);
    }
    G = std::max(1, std::min(G, std::max(1, nch)));
    const int cps = (nch + G - 1) / G;  // chunks per segment
    *seg_len = std::max(1, cps) * 64;
    *G_out = nch > 0 ? (nch + cps - 1) / cps : 1;
    return EFLA_OK;
}

static size_t scan_bytes(int B, int H, int d_k, int d_v, int G) {
    return G <= 1 ? 0 : (size_t)(3 * G - 2) * B * H * d_k * d_v * sizeof(float);
}

efla_status efla_fwd_scan_workspace(int B, int T, int H, int d_k, int d_v, int segments, size_t *bytes,
                                    int *segments_used) {
    if (!bytes) return fail(EFLA_ERR_INVALID_ARG, "bytes must be non-NULL");
    if (B < 0 || T < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d", B, T, H);
    int G = 1, seg = 64;
    efla_status s = scan_plan(B, T, H, segments, &G, &seg);
    if (s != EFLA_OK) return s;
    *bytes = scan_bytes(B, H, d_k, d_v, G);
    if (segments_used) *segments_used = G;
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_fwd_chunked_scan(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                                  void *o, float *S_T, int B, int T, int H, int d_k, int d_v, efla_dtype in_dtype,
                                  efla_dtype o_dtype, int segments, void *workspace, size_t workspace_bytes,
                                  efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    FwdArgs a{q, k, v, beta, S0, nullptr, o, S_T, B, T, H, d_k, d_v, B, in_dtype, o_dtype, 64,
              reinterpret_cast<cudaStream_t>(stream), nullptr, (int)update};
    efla_status s = validate_fwd(a, true);
    if (s != EFLA_OK) return s;
    const bool tc = in_dtype == EFLA_BF16 && d_k == 128 && d_v == 128;
    int G = 1, seg = 64;
    if (tc && (long long)B * T > 0) {
        s = scan_plan(B, T, H, segments, &G, &seg);
        if (s != EFLA_OK) return s;
    }
    if (G <= 1) return run_fwd(a, true);  // one segment (or a CUDA-core shape): the plain forward
    const size_t need = scan_bytes(B, H, d_k, d_v, G);
    if (!workspace || workspace_bytes < need)
        return fail(EFLA_ERR_INVALID_ARG, "workspace of %zu bytes needed (%zu given)", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (!aligned16(workspace)) return fail(EFLA_ERR_INVALID_ARG, "workspace=%p is not 16-byte aligned", workspace);
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace);
    const Range ws{"workspace", w0, w0 + need};
    const size_t th = (size_t)B * T * H, st = (size_t)B * H * d_k * d_v * 4;
    auto R = [](const char *n, const void *p, size_t bytes) {
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{n, lo, p ? lo + bytes : lo};
    };
    const Range others[] = {R("q", q, th * d_k * dsize(in_dtype)), R("k", k, th * d_k * dsize(in_dtype)),
                            R("v", v, th * d_v * dsize(in_dtype)), R("beta", beta, th * 4), R("S0", S0, st),
                            R("o", o, th * d_v * dsize(o_dtype)), R("S_T", S_T, st)};
    for (const Range &r : others)
        if (overlap(ws, r)) return fail(EFLA_ERR_INVALID_ARG, "workspace overlaps %s", r.name);
    a.status = device_status_ptr();
    if (!a.status) return fail(EFLA_ERR_CUDA, "cannot resolve the device status word");
    float *s_in = static_cast<float *>(workspace);
    float *maps = s_in + (size_t)G * B * H * d_k * d_v;
    const char *why = nullptr;
    FwdArgs m = a;  // pass 1: the maps of segments 0..G-2 (no outputs)
    m.o = nullptr;
    m.S_T = nullptr;
    m.S0 = nullptr;
    m.seg_len = seg;
    m.G = G;
    m.maps = maps;
    cudaError_t e = launch_chunk_tc(m, &why);
    if (e != cudaSuccess) return cuda_fail(e, why ? why : "segment-map launch");
    e = launch_scan_combine(S0, maps, s_in, B, G, H, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "segment scan launch");
    FwdArgs f = a;  // pass 2: every segment from its start state, with outputs
    f.seg_len = seg;
    f.G = G;
    f.s_in = s_in;
    e = launch_chunk_tc(f, &why);
    if (e != cudaSuccess) return cuda_fail(e, why ? why : "segmented forward launch");
    g_last_error.clear();
    return EFLA_OK;
}

// Device address of the static scratch, resolved once per device.
static void *scan_scratch_ptr() {
    static std::mutex mu;
    static void *ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scan_scratch) == cudaSuccess) ptrs[dev] = p;
    }
    return ptrs[dev];
}

efla_status efla_fwd_chunked_scan_static(const void *q, const void *k, const void *v, const float *beta,
                                         const float *S0, void *o, float *S_T, int B, int T, int H, int d_k,
                                         int d_v, efla_dtype in_dtype, efla_dtype o_dtype, int segments,
                                         efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    if (B < 0 || T < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d", B, T, H);
    size_t need = 0;
    const bool tc = in_dtype == EFLA_BF16 && d_k == 128 && d_v == 128;
    if (tc && (long long)B * T > 0) {
        int G = 1, seg = 64;
        efla_status s = scan_plan(B, T, H, segments, &G, &seg);
        if (s != EFLA_OK) return s;
        need = scan_bytes(B, H, d_k, d_v, G);
        if (segments <= 0) {  // automatic split: the most pieces whose maps and states fit the scratch
            while (G > 1 && need > SCAN_SCRATCH_BYTES) {
                s = scan_plan(B, T, H, G - 1, &G, &seg);
                if (s != EFLA_OK) return s;
                need = scan_bytes(B, H, d_k, d_v, G);
            }
            segments = G;
        }
    }
    if (need > SCAN_SCRATCH_BYTES)
        return fail(EFLA_ERR_UNSUPPORTED, "this split needs %zu bytes of scratch; the static scratch holds %zu",
                    need, SCAN_SCRATCH_BYTES);
    void *ws = nullptr;
    if (need > 0 && !(ws = scan_scratch_ptr())) return fail(EFLA_ERR_CUDA, "cannot resolve the static scratch");
    // Nothing in the scratch has to start at zero: every state and map is written before it is read.
    return efla_fwd_chunked_scan(q, k, v, beta, S0, o, S_T, B, T, H, d_k, d_v, in_dtype, o_dtype, segments, ws,
                                 need > 0 ? SCAN_SCRATCH_BYTES : 0, update, stream);
}

efla_status efla_bwd_recurrent(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                               const float *dO, const float *dS_T, float *dq, float *dk, float *dv, float *dbeta,
                               float *dS0, int B, int T, int H, int d_k, int d_v, efla_dtype in_dtype,
                               efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    if (B < 0 || T < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d", B, T, H);
    efla_status s = check_dims_common(d_k, d_v, in_dtype, EFLA_F32);
    if (s != EFLA_OK) return s;
    const long long rows = (long long)B * T * H;
    if (rows > (1LL << 31) - 1) return fail(EFLA_ERR_UNSUPPORTED, "B*T*H=%lld exceeds 2^31-1", rows);
    if (rows > 0 && (!q || !k || !v || !beta || !dO || !dq || !dk || !dv || !dbeta))
        return fail(EFLA_ERR_INVALID_ARG, "q, k, v, beta, dO, dq, dk, dv and dbeta must be non-NULL when B*T > 0");
    const void *ptrs[] = {q, k, v, beta, S0, dO, dS_T, dq, dk, dv, dbeta, dS0};
    const char *names[] = {"q", "k", "v", "beta", "S0", "dO", "dS_T", "dq", "dk", "dv", "dbeta", "dS0"};
    for (int i = 0; i < 12; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(EFLA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    const size_t th = (size_t)rows, st = (size_t)B * H * d_k * d_v * 4;
    auto R = [](const char *n, const void *p, size_t bytes) {
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{n, lo, p ? lo + bytes : lo};
    };
    const Range in[] = {R("q", q, th * d_k * dsize(in_dtype)), R("k", k, th * d_k * dsize(in_dtype)),
                        R("v", v, th * d_v * dsize(in_dtype)), R("beta", beta, th * 4), R("S0", S0, st),
                        R("dO", dO, th * d_v * 4), R("dS_T", dS_T, st)};
    const Range out[] = {R("dq", dq, th * d_k * 4), R("dk", dk, th * d_k * 4), R("dv", dv, th * d_v * 4),
                         R("dbeta", dbeta, th * 4), R("dS0", dS0, st)};
    for (int i = 0; i < 5; ++i) {
        for (const Range &r : in)
            if (overlap(out[i], r)) return fail(EFLA_ERR_INVALID_ARG, "output %s overlaps input %s", out[i].name, r.name);
        for (int j = i + 1; j < 5; ++j)
            if (overlap(out[i], out[j])) return fail(EFLA_ERR_INVALID_ARG, "outputs %s and %s overlap", out[i].name, out[j].name);
    }
    BwdArgs a{q, k, v, beta, S0, dO, dS_T, dq, dk, dv, dbeta, dS0, B, T, H, d_k, d_v, in_dtype,
              reinterpret_cast<cudaStream_t>(stream), (int)update};
    cudaError_t e = launch_bwd(a);
    if (e != cudaSuccess) return cuda_fail(e, "backward kernel launch");
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_bwd_workspace(int B, int T, int H, int d_k, int d_v, size_t *bytes) {
    if (!bytes) return fail(EFLA_ERR_INVALID_ARG, "bytes must be non-NULL");
    if (B < 0 || T < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d", B, T, H);
    if (d_k != d_v || (d_k != 64 && d_k != 128))
        return fail(EFLA_ERR_UNSUPPORTED, "the chunked backward supports d_k = d_v in {64, 128} (got %d, %d)", d_k, d_v);
    const size_t nc = ((size_t)T + 63) / 64;
    // per chunk: start state and end-state gradient (4 bytes an element), T'' (64 x 64 x 4 bytes);
    // per token: dO as bf16 hi and lo, G (fp32), -dR as bf16 hi and lo
    *bytes = (size_t)B * H * nc * (2 * (size_t)d_k * d_v + 64 * 64) * sizeof(float) +
             (size_t)B * T * H * d_v * (2 * 2 + sizeof(float) + 2 * 2);
    return EFLA_OK;
}

// The chunked backward; with `saved`, the workspace already holds the chunk-start states and T''
// tiles of this forward (efla_fwd_chunked_train) and the forward is not run again.
static efla_status bwd_chunked_impl(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                                    const float *dO, const float *dS_T, float *dq, float *dk, float *dv, float *dbeta,
                                    float *dS0, int B, int T, int H, int d_k, int d_v, efla_dtype in_dtype,
                                    efla_update update, void *workspace, size_t workspace_bytes, efla_stream_t stream,
                                    bool saved) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    if (B < 0 || T < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d", B, T, H);
    efla_status s = check_dims_common(d_k, d_v, in_dtype, EFLA_F32);
    if (s != EFLA_OK) return s;
    size_t need = 0;
    if ((s = efla_bwd_workspace(B, T, H, d_k, d_v, &need)) != EFLA_OK) return s;
    const long long rows = (long long)B * T * H;
    if (rows > (1LL << 31) - 1) return fail(EFLA_ERR_UNSUPPORTED, "B*T*H=%lld exceeds 2^31-1", rows);
    if (rows > 0 && (!q || !k || !v || !beta || !dO || !dq || !dk || !dv || !dbeta))
        return fail(EFLA_ERR_INVALID_ARG, "q, k, v, beta, dO, dq, dk, dv and dbeta must be non-NULL when B*T > 0");
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(EFLA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu at %p)", need, workspace_bytes,
                    workspace);
    const void *ptrs[] = {q, k, v, beta, S0, dO, dS_T, dq, dk, dv, dbeta, dS0, workspace};
    const char *names[] = {"q", "k", "v", "beta", "S0", "dO", "dS_T", "dq", "dk", "dv", "dbeta", "dS0", "workspace"};
    for (int i = 0; i < 13; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(EFLA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    const size_t th = (size_t)rows, st = (size_t)B * H * d_k * d_v * 4;
    auto R = [](const char *n, const void *p, size_t bytes) {
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{n, lo, p ? lo + bytes : lo};
    };
    const Range in[] = {R("q", q, th * d_k * dsize(in_dtype)), R("k", k, th * d_k * dsize(in_dtype)),
                        R("v", v, th * d_v * dsize(in_dtype)), R("beta", beta, th * 4), R("S0", S0, st),
                        R("dO", dO, th * d_v * 4), R("dS_T", dS_T, st)};
    const Range out[] = {R("dq", dq, th * d_k * 4), R("dk", dk, th * d_k * 4), R("dv", dv, th * d_v * 4),
                         R("dbeta", dbeta, th * 4), R("dS0", dS0, st), R("workspace", workspace, need)};
    for (int i = 0; i < 6; ++i) {
        for (const Range &r : in)
            if (overlap(out[i], r)) return fail(EFLA_ERR_INVALID_ARG, "%s overlaps input %s", out[i].name, r.name);
        for (int j = i + 1; j < 6; ++j)
            if (overlap(out[i], out[j])) return fail(EFLA_ERR_INVALID_ARG, "%s and %s overlap", out[i].name, out[j].name);
    }
    if ((long long)B * H == 0) {
        g_last_error.clear();
        return EFLA_OK;
    }
    int *status = device_status_ptr();
    if (!status) return fail(EFLA_ERR_CUDA, "cannot resolve the device status word");
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t state_floats = (size_t)B * H * (((size_t)T + 63) / 64) * d_k * d_v;
    float *states = static_cast<float *>(workspace);
    float *dse = states + state_floats;
    uint8_t *tpp = reinterpret_cast<uint8_t *>(dse + state_floats);
    void *do_split = tpp + (size_t)B * H * (((size_t)T + 63) / 64) * 64 * 64 * 4;
    float *g_tok = reinterpret_cast<float *>(static_cast<char *>(do_split) + 2 * (size_t)B * T * H * d_v * 2);
    void *dr_split = g_tok + (size_t)B * T * H * d_v;
    cudaError_t e;
    if (T > 0 && !saved) {  // the forward, keeping the state at the start of every chunk (o and S_T not needed)
        FwdArgs fa{q, k, v, beta, S0, nullptr, nullptr, nullptr, B, T, H, d_k, d_v, B, in_dtype, in_dtype,
                   64, cs, status, (int)update};
        fa.states = states;
        fa.tpp = tpp;
        const char *why = "chunk kernel launch (backward states)";
        e = in_dtype == EFLA_BF16 && d_k == 128 ? launch_chunk_tc(fa, &why) : launch_chunk_simt(fa);
        if (e != cudaSuccess) return cuda_fail(e, why);
    }
    BwdArgs a{q, k, v, beta, S0, dO, dS_T, dq, dk, dv, dbeta, dS0, B, T, H, d_k, d_v, in_dtype, cs, (int)update};
    const bool tc = in_dtype == EFLA_BF16 && d_k == 128 && T > 0;  // the state pass on the tensor cores
    if (tc) {
        const char *why = "tcgen05 state-gradient kernel launch";
        e = launch_bwd_state_tc(a, dse, tpp, do_split, g_tok, dr_split, &why);
        if (e == cudaSuccess) e = launch_bwd_grad_tc(a, states, dse, tpp, do_split, g_tok, dr_split, &why);
        if (e != cudaSuccess) return cuda_fail(e, why);
    } else {
        e = launch_bwd_chunked(a, states, dse);
        if (e != cudaSuccess) return cuda_fail(e, "chunked backward kernel launch");
    }
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_bwd_chunked(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                             const float *dO, const float *dS_T, float *dq, float *dk, float *dv, float *dbeta,
                             float *dS0, int B, int T, int H, int d_k, int d_v, efla_dtype in_dtype,
                             efla_update update, void *workspace, size_t workspace_bytes, efla_stream_t stream) {
    return bwd_chunked_impl(q, k, v, beta, S0, dO, dS_T, dq, dk, dv, dbeta, dS0, B, T, H, d_k, d_v, in_dtype, update,
                            workspace, workspace_bytes, stream, false);
}

efla_status efla_bwd_chunked_saved(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                                   const float *dO, const float *dS_T, float *dq, float *dk, float *dv,
                                   float *dbeta, float *dS0, int B, int T, int H, int d_k, int d_v,
                                   efla_dtype in_dtype, efla_update update, void *workspace, size_t workspace_bytes,
                                   efla_stream_t stream) {
    return bwd_chunked_impl(q, k, v, beta, S0, dO, dS_T, dq, dk, dv, dbeta, dS0, B, T, H, d_k, d_v, in_dtype, update,
                            workspace, workspace_bytes, stream, true);
}

efla_status efla_fwd_chunked_train(const void *q, const void *k, const void *v, const float *beta, const float *S0,
                                   void *o, float *S_T, int B, int T, int H, int d_k, int d_v, efla_dtype in_dtype,
                                   efla_update update, void *workspace, size_t workspace_bytes,
                                   efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    FwdArgs a{q, k, v, beta, S0, nullptr, o, S_T, B, T, H, d_k, d_v, B, in_dtype, in_dtype, 64,
              reinterpret_cast<cudaStream_t>(stream), nullptr, (int)update};
    efla_status s = validate_fwd(a, true);
    if (s != EFLA_OK) return s;
    size_t need = 0;
    if ((s = efla_bwd_workspace(B, T, H, d_k, d_v, &need)) != EFLA_OK) return s;
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(EFLA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu at %p)", need, workspace_bytes,
                    workspace);
    if (workspace && !aligned16(workspace))
        return fail(EFLA_ERR_INVALID_ARG, "workspace=%p is not 16-byte aligned", workspace);
    const size_t th = (size_t)B * T * H, st = (size_t)B * H * d_k * d_v * 4;
    auto R = [](const char *n, const void *p, size_t bytes) {
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{n, lo, p ? lo + bytes : lo};
    };
    const Range ws = R("workspace", workspace, need);
    const Range others[] = {R("q", q, th * d_k * dsize(in_dtype)), R("k", k, th * d_k * dsize(in_dtype)),
                            R("v", v, th * d_v * dsize(in_dtype)), R("beta", beta, th * 4), R("S0", S0, st),
                            R("o", o, th * d_v * dsize(in_dtype)), R("S_T", S_T, st)};
    for (const Range &r : others)
        if (overlap(ws, r)) return fail(EFLA_ERR_INVALID_ARG, "workspace overlaps %s", r.name);
    if ((long long)B * H == 0 || T == 0) return run_fwd(a, true);
    a.status = device_status_ptr();
    if (!a.status) return fail(EFLA_ERR_CUDA, "cannot resolve the device status word");
    const size_t state_floats = (size_t)B * H * (((size_t)T + 63) / 64) * d_k * d_v;
    a.states = static_cast<float *>(workspace);
    a.tpp = reinterpret_cast<uint8_t *>(a.states + 2 * state_floats);  // the layout efla_bwd_chunked uses
    cudaError_t e;
    const char *why = "chunk kernel launch (training forward)";
    e = in_dtype == EFLA_BF16 && d_k == 128 ? launch_chunk_tc(a, &why) : launch_chunk_simt(a);
    if (e != cudaSuccess) return cuda_fail(e, why);
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_fwd_recurrent_ex(const void *q, const void *k, const void *v, const float *beta,
                                  const float *S0, const int32_t *cu_seqlens, void *o, float *S_T, int B,
                                  int T, int H, int d_k, int d_v, int N, efla_dtype in_dtype,
                                  efla_dtype o_dtype, efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    FwdArgs a{q, k, v, beta, S0, cu_seqlens, o, S_T, B, T, H, d_k, d_v, N, in_dtype, o_dtype,
              0, reinterpret_cast<cudaStream_t>(stream), nullptr, (int)update};
    return run_fwd(a, false);
}

efla_status efla_fwd_recurrent(const void *q, const void *k, const void *v, const float *beta,
                               const float *S0, const int32_t *cu_seqlens, void *o, float *S_T, int B,
                               int T, int H, int d_k, int d_v, int N, efla_dtype dtype, efla_stream_t stream) {
    return efla_fwd_recurrent_ex(q, k, v, beta, S0, cu_seqlens, o, S_T, B, T, H, d_k, d_v, N, dtype, dtype,
                                 EFLA_UPDATE_EXACT, stream);
}

efla_status efla_decode_step_ex(const void *q, const void *k, const void *v, const float *beta, float *S,
                                void *o, int B, int H, int d_k, int d_v, efla_dtype in_dtype,
                                efla_dtype o_dtype, efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    if (B < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d H=%d", B, H);
    efla_status s = check_dims_common(d_k, d_v, in_dtype, o_dtype);
    if (s != EFLA_OK) return s;
    if ((long long)B * H > (1LL << 31) - 1) return fail(EFLA_ERR_UNSUPPORTED, "B*H too large");
    if (B > 0 && (!q || !k || !v || !beta || !S || !o))
        return fail(EFLA_ERR_INVALID_ARG, "q, k, v, beta, S and o must be non-NULL when B > 0");
    const void *ptrs[] = {q, k, v, beta, S, o};
    const char *names[] = {"q", "k", "v", "beta", "S", "o"};
    for (int i = 0; i < 6; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(EFLA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    const size_t u = (size_t)B * H;
    auto rng = [](const void *p, size_t n) {
        return Range{"", reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + n};
    };
    const Range rS = rng(S, u * d_k * d_v * 4), ro = rng(o, u * d_v * dsize(o_dtype));
    const Range ins[] = {rng(q, u * d_k * dsize(in_dtype)), rng(k, u * d_k * dsize(in_dtype)),
                         rng(v, u * d_v * dsize(in_dtype)), rng(beta, u * 4)};
    for (const Range &r : ins)
        if (overlap(rS, r) || overlap(ro, r)) return fail(EFLA_ERR_INVALID_ARG, "an output overlaps an input");
    if (overlap(rS, ro)) return fail(EFLA_ERR_INVALID_ARG, "o overlaps S");
    DecodeArgs a{q, k, v, beta, S, o, B, H, d_k, d_v, in_dtype, o_dtype, reinterpret_cast<cudaStream_t>(stream),
                 (int)update};
    cudaError_t e = launch_decode(a);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_decode_step(const void *q, const void *k, const void *v, const float *beta, float *S, void *o,
                             int B, int H, int d_k, int d_v, efla_dtype dtype, efla_stream_t stream) {
    return efla_decode_step_ex(q, k, v, beta, S, o, B, H, d_k, d_v, dtype, dtype, EFLA_UPDATE_EXACT, stream);
}

efla_status efla_decode_tokens(const void *q, const void *k, const void *v, const float *beta, float *S, void *o,
                               int B, int m, int H, int d_k, int d_v, efla_dtype in_dtype, efla_dtype o_dtype,
                               efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    if (B < 0 || m < 0 || H <= 0) return fail(EFLA_ERR_INVALID_ARG, "bad sizes B=%d m=%d H=%d", B, m, H);
    efla_status s = check_dims_common(d_k, d_v, in_dtype, o_dtype);
    if (s != EFLA_OK) return s;
    if ((long long)B * H > (1LL << 31) - 1 || (long long)B * m * H > (1LL << 40))
        return fail(EFLA_ERR_UNSUPPORTED, "B*H or B*m*H too large");
    if (B > 0 && !S) return fail(EFLA_ERR_INVALID_ARG, "S must be non-NULL when B > 0");
    if (B > 0 && m > 0 && (!q || !k || !v || !beta || !o))
        return fail(EFLA_ERR_INVALID_ARG, "q, k, v, beta and o must be non-NULL when B*m > 0");
    const void *ptrs[] = {q, k, v, beta, S, o};
    const char *names[] = {"q", "k", "v", "beta", "S", "o"};
    for (int i = 0; i < 6; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(EFLA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    const size_t u = (size_t)B * H, rows = (size_t)B * m * H;
    auto rng = [](const void *p, size_t n) {
        return Range{"", reinterpret_cast<uintptr_t>(p), p ? reinterpret_cast<uintptr_t>(p) + n : 0};
    };
    const Range rS = rng(S, u * d_k * d_v * 4), ro = rng(o, rows * d_v * dsize(o_dtype));
    const Range ins[] = {rng(q, rows * d_k * dsize(in_dtype)), rng(k, rows * d_k * dsize(in_dtype)),
                         rng(v, rows * d_v * dsize(in_dtype)), rng(beta, rows * 4)};
    for (const Range &r : ins)
        if (overlap(rS, r) || overlap(ro, r)) return fail(EFLA_ERR_INVALID_ARG, "an output overlaps an input");
    if (overlap(rS, ro)) return fail(EFLA_ERR_INVALID_ARG, "o overlaps S");
    DecodeArgs a{q, k, v, beta, S, o, B, H, d_k, d_v, in_dtype, o_dtype, reinterpret_cast<cudaStream_t>(stream),
                 (int)update, m};
    const char *why = "decode-tokens kernel launch";
    cudaError_t e = in_dtype == EFLA_BF16 && d_k == 128 && d_v == 128 ? launch_decode_tokens_tc(a, &why)
                                                                       : launch_decode_tokens(a);
    if (e != cudaSuccess) return cuda_fail(e, why);
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_prep(const void *k, const void *v, const float *beta, float *lam, float *alpha, void *ak, void *av,
                      long long n, int d_k, int d_v, efla_dtype dtype, efla_update update, efla_stream_t stream) {
    if (!update_ok(update)) return fail(EFLA_ERR_INVALID_ARG, "unknown update rule %d", (int)update);
    if (n < 0) return fail(EFLA_ERR_INVALID_ARG, "n=%lld must be >= 0", n);
    efla_status s = check_dims_common(d_k, d_v, dtype, dtype);
    if (s != EFLA_OK) return s;
    if (n > (1LL << 40)) return fail(EFLA_ERR_UNSUPPORTED, "n=%lld too large", n);
    if (n > 0 && (!k || !beta)) return fail(EFLA_ERR_INVALID_ARG, "k and beta must be non-NULL when n > 0");
    if (n > 0 && av && !v) return fail(EFLA_ERR_INVALID_ARG, "v must be non-NULL when av is requested");
    const void *ptrs[] = {k, v, beta, lam, alpha, ak, av};
    const char *names[] = {"k", "v", "beta", "lam", "alpha", "ak", "av"};
    for (int i = 0; i < 7; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(EFLA_ERR_INVALID_ARG, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    auto R = [](const char *nm, const void *p, size_t bytes) {
        uintptr_t lo = reinterpret_cast<uintptr_t>(p);
        return Range{nm, lo, p ? lo + bytes : lo};
    };
    const size_t un = (size_t)n;
    const Range in[] = {R("k", k, un * d_k * dsize(dtype)), R("v", av ? v : nullptr, un * d_v * dsize(dtype)),
                        R("beta", beta, un * 4)};
    const Range out[] = {R("lam", lam, un * 4), R("alpha", alpha, un * 4), R("ak", ak, un * d_k * dsize(dtype)),
                         R("av", av, un * d_v * dsize(dtype))};
    for (int i = 0; i < 4; ++i) {
        for (const Range &r : in)
            if (overlap(out[i], r)) return fail(EFLA_ERR_INVALID_ARG, "output %s overlaps input %s", out[i].name, r.name);
        for (int j = i + 1; j < 4; ++j)
            if (overlap(out[i], out[j])) return fail(EFLA_ERR_INVALID_ARG, "outputs %s and %s overlap", out[i].name, out[j].name);
    }
    PrepArgs a{k, av ? v : nullptr, beta, lam, alpha, ak, av, n, d_k, d_v, dtype, (int)update,
               reinterpret_cast<cudaStream_t>(stream)};
    cudaError_t e = launch_prep(a);
    if (e != cudaSuccess) return cuda_fail(e, "prep kernel launch");
    g_last_error.clear();
    return EFLA_OK;
}

efla_status efla_device_status(efla_stream_t stream) {
    int *p = device_status_ptr();
    if (!p) return fail(EFLA_ERR_CUDA, "cannot resolve the device status word");
    int h = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, p, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (h != EFLA_OK) {
        g_last_error = h == EFLA_ERR_DEVICE_TIMEOUT ? "a bounded in-kernel wait expired"
                       : h == EFLA_ERR_INVALID_ARG  ? "a kernel met malformed cu_seqlens bounds"
                                                     : "a kernel recorded an error";
        return static_cast<efla_status>(h);
    }
    return EFLA_OK;
}

const char *efla_get_error_string(efla_status s) {
    switch (s) {
        case EFLA_OK: return "EFLA_OK";
        case EFLA_ERR_INVALID_ARG: return "EFLA_ERR_INVALID_ARG: invalid argument";
        case EFLA_ERR_UNSUPPORTED: return "EFLA_ERR_UNSUPPORTED: valid but unsupported configuration";
        case EFLA_ERR_CUDA: return "EFLA_ERR_CUDA: CUDA call or kernel launch failed";
        case EFLA_ERR_DEVICE_TIMEOUT: return "EFLA_ERR_DEVICE_TIMEOUT: a bounded in-kernel wait expired";
    }
    return "unknown efla_status";
}

void efla_debug_set_wait_limit_ns(unsigned long long ns) { set_wait_limit_ns(ns); }

void efla_debug_set_stall(int stall) { g_debug_stall.store(stall & 7, std::memory_order_relaxed); }

const char *efla_last_error(void) { return g_last_error.c_str(); }

int efla_abi_version(void) { return EFLA_ABI_VERSION; }

}  // extern "C"
