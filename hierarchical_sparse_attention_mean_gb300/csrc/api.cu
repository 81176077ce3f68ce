// api.cu -- the C ABI of include/llsa.h: parameter validation, size
// derivation, workspace checks, device checks, status word and launch
// accounting. Every compute step runs in the kernels of the other units.
#include <math.h>
#include <string.h>

#include <atomic>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"
#include "tc.cuh"

namespace llsa {

// ----------------------------------------------------------- status word --

static __device__ int g_status;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_addr[kMaxDevices];
int g_sm_count[kMaxDevices];
int g_cc_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 wrong device
std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_wait_limit{0};  // 0: the kernels' own limit
std::atomic<int> g_test_flags{0};

struct ProfRecord {
    const char* name;
    cudaEvent_t start, stop;
};
bool g_prof_on = false;
std::string g_prof_prefix;            // record only launches whose name starts with it ("" : all)
thread_local bool t_prof_open = false;  // launch_begin recorded a start event for this thread's launch
std::vector<ProfRecord> g_prof;
std::vector<cudaEvent_t> g_event_pool;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Compute capability 10.3 (GB300) is the only target of this library.
int check_device() {
    int dev = current_device();
    if (dev < 0) return LLSA_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            return LLSA_ERR_DEVICE;
        }
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_sm_count[dev] = sms;
        void* addr = nullptr;
        if (g_cc_ok[dev] == 1) {
            if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) {
                g_cc_ok[dev] = 0;
                return LLSA_ERR_CUDA;
            }
            g_status_addr[dev] = static_cast<int*>(addr);
        }
    }
    return g_cc_ok[dev] == 1 ? LLSA_OK : LLSA_ERR_DEVICE;
}

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

int device_ready() { return check_device(); }

int* status_ptr() {
    int dev = current_device();
    return dev < 0 ? nullptr : g_status_addr[dev];
}

int sm_count() {
    int dev = current_device();
    return (dev < 0 || g_sm_count[dev] <= 0) ? 148 : g_sm_count[dev];
}

void launch_begin(const char* name, cudaStream_t st) {
    t_prof_open = false;
    if (!g_prof_on) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_prof_prefix.empty() && strncmp(name, g_prof_prefix.c_str(), g_prof_prefix.size()) != 0) return;
    t_prof_open = true;
    ProfRecord r{name, take_event(), take_event()};
    cudaEventRecord(r.start, st);
    g_prof.push_back(r);
}

int launch_end(const char* name, cudaStream_t st) {
    (void)name;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (t_prof_open) {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_prof.empty()) cudaEventRecord(g_prof.back().stop, st);
        t_prof_open = false;
    }
    return cudaGetLastError() == cudaSuccess ? LLSA_OK : LLSA_ERR_CUDA;
}

// ------------------------------------------------------------ validation --

static int derive(const llsa_params* p, Shape* s) {
    if (!p) return LLSA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->heads < 0 || p->n < 1 || p->topk < 1) return LLSA_ERR_INVALID_ARG;
    if (p->dtype != LLSA_DTYPE_BF16 && p->dtype != LLSA_DTYPE_F32) return LLSA_ERR_DTYPE;
    if (p->enrich_rule != LLSA_ENRICH_TOP1 && p->enrich_rule != LLSA_ENRICH_ANCESTOR &&
        p->enrich_rule != LLSA_ENRICH_ALLK)
        return LLSA_ERR_INVALID_ARG;
    if (!(p->scale >= 0.0f) || isinf(p->scale)) return LLSA_ERR_INVALID_ARG;
    if (p->token_order != LLSA_ORDER_TILE && p->token_order != LLSA_ORDER_RASTER) return LLSA_ERR_INVALID_ARG;
    if (p->d < 8 || p->d > 256 || p->d % 8 != 0) return LLSA_ERR_SHAPE;
    if (p->block < 2 || p->block > 1024) return LLSA_ERR_SHAPE;
    const long long n = p->n, B = p->block;
    // L_max = floor(log_B n - 1) = (largest e with B^e <= n) - 1
    int e = 0;
    long long pw = 1;
    while (pw * B <= n) { pw *= B; e++; }
    int Lmax = e - 1;
    if (Lmax < 1) return LLSA_ERR_SHAPE;
    int L = p->levels == 0 ? Lmax : p->levels;
    if (L < 1 || L > Lmax) return LLSA_ERR_SHAPE;
    if (L > LLSA_MAX_LEVELS) return LLSA_ERR_UNSUPPORTED;
    memset(s, 0, sizeof(*s));
    s->n_level[0] = p->n;
    for (int l = 1; l <= L; l++) {
        if (s->n_level[l - 1] % p->block != 0) return LLSA_ERR_SHAPE;
        s->n_level[l] = s->n_level[l - 1] / p->block;
    }
    int Le = p->enrich_levels < 0 ? L : p->enrich_levels;
    if (Le > L) return LLSA_ERR_SHAPE;
    // K clamped to the candidates of each level
    long long c = s->n_level[L];
    s->topk_level[L] = (int)(p->topk < c ? p->topk : c);
    for (int l = L - 1; l >= 1; l--) {
        c = (long long)s->topk_level[l + 1] * p->block;
        s->topk_level[l] = (int)(p->topk < c ? p->topk : c);
    }
    int off = 0;
    for (int l = 1; l <= L; l++) { s->row_offset[l] = off; off += s->n_level[l]; }
    long long lio = 0;
    for (int l = 2; l <= L; l++) {
        s->level_idx_offset[l] = lio;
        lio += (long long)s->n_level[l] * s->topk_level[l];
    }
    s->level_idx_per_slice = lio;
    s->slices = (long long)p->batch * p->heads;
    s->n = p->n; s->d = p->d; s->B = p->block; s->L = L; s->Le = Le; s->rule = p->enrich_rule; s->topk = p->topk;
    s->K1 = s->topk_level[1]; s->T = s->n_level[1]; s->P = off; s->dtype = p->dtype;
    // enrichment columns: one per level, or K_l per level under ALLK
    s->col_off[1] = 0;
    for (int l = 1; l <= L; l++)
        s->col_off[l + 1] = s->col_off[l] + (p->enrich_rule == LLSA_ENRICH_ALLK ? s->topk_level[l] : 1);
    s->C = s->col_off[L + 1];
    s->Lc = s->col_off[Le + 1];
    if (s->Lc > kMaxCoarse) return LLSA_ERR_UNSUPPORTED;
    s->scale = p->scale > 0.0f ? p->scale : 1.0f / sqrtf((float)p->d);
    if (s->slices * (long long)p->n * p->d > (1LL << 40)) return LLSA_ERR_UNSUPPORTED;
    if (p->token_order == LLSA_ORDER_RASTER) {
        // a square image of side 4^m, blocks of 4 x 4 tokens
        int side = 1;
        while ((long long)side * side < p->n) side *= 4;
        if (p->block != 16 || (long long)side * side != p->n || side < 4) return LLSA_ERR_SHAPE;
        s->raster = 1;
        s->side = side;
    }
    return LLSA_OK;
}

static bool aligned(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

static int check_ptrs(std::initializer_list<const void*> ptrs) {
    for (const void* q : ptrs) {
        if (!q) return LLSA_ERR_INVALID_ARG;
        if (!aligned(q)) return LLSA_ERR_ALIGN;
    }
    return LLSA_OK;
}

static size_t transpose_ws(const Shape& s) { return (size_t)s.slices * s.T * sizeof(int32_t); }

// An NVTX range around a C-ABI call (the call's name), so a profiler timeline
// shows each library call with the kernels it enqueued.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
};

int wait_limit() {
    const int v = g_wait_limit.load();
    return v > 0 ? v : tc::kSpinLimit;
}

int test_flags() { return g_test_flags.load(); }

}  // namespace llsa

using namespace llsa;

extern "C" {

int llsa_test_set_wait_limit(int polls, int flags) {
    if (flags & ~(LLSA_TEST_NO_COPIES | LLSA_TEST_FORCE_GROUPED | LLSA_TEST_FORCE_PER_BLOCK)) return LLSA_ERR_INVALID_ARG;
    if ((flags & LLSA_TEST_FORCE_GROUPED) && (flags & LLSA_TEST_FORCE_PER_BLOCK)) return LLSA_ERR_INVALID_ARG;
    g_wait_limit.store(polls > 0 ? polls : 0);
    g_test_flags.store(flags);
    return LLSA_OK;
}

int llsa_get_sizes(const llsa_params* p, llsa_sizes* out) {
    Shape s;
    if (!out) return LLSA_ERR_INVALID_ARG;
    LLSA_TRY(derive(p, &s));
    memset(out, 0, sizeof(*out));
    out->levels = s.L;
    out->enrich_levels = s.Le;
    for (int l = 0; l <= LLSA_MAX_LEVELS; l++) {
        out->n_level[l] = s.n_level[l];
        out->topk_level[l] = s.topk_level[l];
        out->row_offset[l] = s.row_offset[l];
        out->level_idx_offset[l] = s.level_idx_offset[l];
    }
    out->pyr_rows = s.P;
    out->n_blocks = s.T;
    out->keys_per_query = s.K1 * s.B + s.Lc;
    out->coarse_cols = s.C;
    out->enrich_cols = s.Lc;
    out->slices = s.slices;
    out->level_idx_per_slice = s.level_idx_per_slice;
    out->scale = s.scale;
    return LLSA_OK;
}

size_t llsa_workspace_bytes(const llsa_params* p, int op) {
    Shape s;
    if (derive(p, &s) != LLSA_OK) return 0;
    switch (op) {
        case LLSA_OP_FWD: return fwd_workspace_bytes(s);
        case LLSA_OP_TRANSPOSE: return transpose_ws(s);
        case LLSA_OP_BWD: return bwd_workspace_bytes(s);
        default: return 0;
    }
}

int llsa_pool(const llsa_params* p, const void* q, const void* k, const void* v, float* pyr, void* ws,
              size_t ws_bytes, void* stream) {
    CallRange range("llsa_pool");
    (void)ws; (void)ws_bytes;
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({q, k, v, pyr}));
    LLSA_TRY(check_device());
    return launch_pool(s, q, k, v, pyr, static_cast<cudaStream_t>(stream));
}

int llsa_select_exhaustive(const llsa_params* p, const float* pyr, int32_t* sel_idx, void* stream) {
    CallRange range("llsa_select_exhaustive");
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({pyr, sel_idx}));
    LLSA_TRY(check_device());
    return launch_select_exhaustive(s, pyr, sel_idx, static_cast<cudaStream_t>(stream));
}

int llsa_reorder(const llsa_params* p, int height, int width, const void* in, void* out, int inverse, void* stream) {
    CallRange range("llsa_reorder");
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (inverse != 0 && inverse != 1) return LLSA_ERR_INVALID_ARG;
    int root = 2;
    while (root * root < s.B) root++;
    if (root * root != s.B) return LLSA_ERR_SHAPE;
    if (height != width || height < 1 || (long long)height * width != s.n) return LLSA_ERR_SHAPE;
    int digits = 0;
    for (int side = height; side > 1; side /= root) {
        if (side % root != 0) return LLSA_ERR_SHAPE;
        digits++;
    }
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({in, out}));
    if (in == out) return LLSA_ERR_INVALID_ARG;
    LLSA_TRY(check_device());
    return launch_reorder(s, width, root, digits, in, out, inverse, static_cast<cudaStream_t>(stream));
}

int llsa_select(const llsa_params* p, const float* pyr, int32_t* sel_idx, int32_t* coarse_idx,
                int32_t* level_idx, void* ws, size_t ws_bytes, void* stream) {
    CallRange range("llsa_select");
    (void)ws; (void)ws_bytes;
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({pyr, sel_idx, coarse_idx}));
    if (s.L >= 2) LLSA_TRY(check_ptrs({level_idx}));
    LLSA_TRY(check_device());
    return launch_select(s, pyr, sel_idx, coarse_idx, level_idx, static_cast<cudaStream_t>(stream));
}

int llsa_fwd(const llsa_params* p, const void* q, const void* k, const void* v, const float* pyr,
             const int32_t* sel_idx, const int32_t* coarse_idx, void* o, float* lse, void* ws, size_t ws_bytes,
             void* stream) {
    CallRange range("llsa_fwd");
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({q, k, v, pyr, sel_idx, coarse_idx, o, lse}));
    const size_t need = fwd_workspace_bytes(s);
    if (need > 0 && (!ws || ws_bytes < need)) return LLSA_ERR_WORKSPACE;
    if (need > 0) LLSA_TRY(check_ptrs({ws}));
    LLSA_TRY(check_device());
    return launch_fwd(s, q, k, v, pyr, sel_idx, coarse_idx, o, lse, ws, static_cast<cudaStream_t>(stream));
}

int llsa_index_transpose(const llsa_params* p, const int32_t* sel_idx, int32_t* col_ptr, int32_t* row_idx,
                         void* ws, size_t ws_bytes, void* stream) {
    CallRange range("llsa_index_transpose");
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({sel_idx, col_ptr, row_idx}));
    if (!ws || ws_bytes < transpose_ws(s)) return LLSA_ERR_WORKSPACE;
    LLSA_TRY(check_ptrs({ws}));
    LLSA_TRY(check_device());
    return launch_transpose(s, sel_idx, s.T, s.K1, s.T, col_ptr, row_idx, static_cast<int32_t*>(ws),
                            static_cast<cudaStream_t>(stream));
}

int llsa_bwd(const llsa_params* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, const float* pyr, const int32_t* sel_idx, const int32_t* coarse_idx,
             const int32_t* col_ptr, const int32_t* row_idx, void* dq, void* dk, void* dv, void* ws,
             size_t ws_bytes, void* stream) {
    CallRange range("llsa_bwd");
    Shape s;
    LLSA_TRY(derive(p, &s));
    if (s.slices == 0) return LLSA_OK;
    LLSA_TRY(check_ptrs({q, k, v, o, lse, dout, pyr, sel_idx, coarse_idx, col_ptr, row_idx, dq, dk, dv}));
    size_t need = bwd_workspace_bytes(s);
    if (need > 0 && (!ws || ws_bytes < need)) return LLSA_ERR_WORKSPACE;
    if (need > 0) LLSA_TRY(check_ptrs({ws}));
    LLSA_TRY(check_device());
    return launch_bwd(s, q, k, v, o, lse, dout, pyr, sel_idx, coarse_idx, col_ptr, row_idx, dq, dk, dv, ws,
                      static_cast<cudaStream_t>(stream));
}

int llsa_get_status(void* stream, int* device_status) {
    if (!device_status) return LLSA_ERR_INVALID_ARG;
    LLSA_TRY(check_device());
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int host = 0, zero = 0;
    int* addr = status_ptr();
    if (cudaMemcpyAsync(&host, addr, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return LLSA_ERR_CUDA;
    if (cudaMemcpyAsync(addr, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess) return LLSA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LLSA_ERR_CUDA;
    *device_status = host;
    return LLSA_OK;
}

const char* llsa_strerror(int code) {
    switch (code) {
        case LLSA_OK: return "ok";
        case LLSA_ERR_INVALID_ARG: return "invalid argument";
        case LLSA_ERR_SHAPE: return "unsupported shape (need N >= B^2, N divisible by B^L, d a multiple of 8 up to 256)";
        case LLSA_ERR_DTYPE: return "unsupported dtype";
        case LLSA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case LLSA_ERR_DEVICE: return "current device is not compute capability 10.3";
        case LLSA_ERR_WORKSPACE: return "workspace missing or too small";
        case LLSA_ERR_CUDA: return "CUDA launch failed";
        case LLSA_ERR_UNSUPPORTED: return "sizes beyond the kernels' limits";
        case LLSA_ERR_TIMEOUT: return "device wait timed out";
        case LLSA_ERR_BAD_INDEX: return "index out of range on the device";
        default: return "unknown error";
    }
}

unsigned long long llsa_launch_count(void) { return g_launches.load(); }

int llsa_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_prof_on = on != 0;
    return LLSA_OK;
}

int llsa_profile_only(const char* prefix) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_prof_prefix = prefix ? prefix : "";
    return LLSA_OK;
}

int llsa_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& r : g_prof) {
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof.clear();
    return LLSA_OK;
}

int llsa_profile_read(const char** names, float* ms, int cap) {
    std::lock_guard<std::mutex> lk(g_mu);
    int n = 0;
    for (auto& r : g_prof) {
        if (n >= cap) break;
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            t = -1.f;
        if (names) names[n] = r.name;
        if (ms) ms[n] = t;
        n++;
    }
    return n;
}

}  // extern "C"
