// Host side of the C ABI declared in include/moe_layer.h: argument checks,
// workspace layout, TMA descriptors and the launch sequence of the layer.
// No allocation, no synchronisation (except moe_read_status), no host read
// of device data.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "moe_internal.h"

namespace moe {

int launch_gemm_l1_fwd(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_l2_fwd(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_l2_dgrad(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_l1_dgrad(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_dw1(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_dw2(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_dw1_mg(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_dw2_mg(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_l1_fwd_mx(const GemmArgs&, const GemmMaps&, int, cudaStream_t);
int launch_gemm_l2_fwd_mx(const GemmArgs&, const GemmMaps&, int, cudaStream_t);

int launch_gemm_raw(int f, const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    switch (f) {
        case L1_FWD: return launch_gemm_l1_fwd(a, m, grid, st);
        case L2_FWD: return launch_gemm_l2_fwd(a, m, grid, st);
        case L2_DGRAD: return launch_gemm_l2_dgrad(a, m, grid, st);
        case L1_DGRAD: return launch_gemm_l1_dgrad(a, m, grid, st);
        case DW1: return launch_gemm_dw1(a, m, grid, st);
        case DW2: return launch_gemm_dw2(a, m, grid, st);
        case DW1_MG: return launch_gemm_dw1_mg(a, m, grid, st);
        case DW2_MG: return launch_gemm_dw2_mg(a, m, grid, st);
        case L1_FWD_MX: return launch_gemm_l1_fwd_mx(a, m, grid, st);
        case L2_FWD_MX: return launch_gemm_l2_fwd_mx(a, m, grid, st);
        default: return (int)cudaErrorInvalidValue;
    }
}

namespace {
const char* const kGemmNames[] = {"gemm_l1_fwd", "gemm_l2_fwd", "gemm_l2_dgrad", "gemm_l1_dgrad",
                                  "gemm_dw1",    "gemm_dw2",    "gemm_dw1_mg",   "gemm_dw2_mg",
                                  "gemm_l1_fwd_fp8", "gemm_l2_fwd_fp8"};
}  // namespace

int launch_gemm(int f, const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    if (grid <= 0) return 0;
    trace_pre(st);
    const int e = launch_gemm_raw(f, a, m, grid, st);
    trace_post(st, kGemmNames[f]);
    return e;
}

namespace {

thread_local std::string g_err;

// ------------------------------------------------------------------ tracing
constexpr int kTraceNames = 4096;
struct Trace {
    void* const* events = nullptr;
    int capacity = 0;
    int n = 0;
    const char* names[kTraceNames];
};
thread_local Trace g_trace;

}  // namespace

void trace_pre(cudaStream_t st) {
    Trace& t = g_trace;
    if (t.events && 2 * t.n + 1 < t.capacity) cudaEventRecord((cudaEvent_t)t.events[2 * t.n], st);
}
void trace_post(cudaStream_t st, const char* name) {
    Trace& t = g_trace;
    if (!t.events) return;
    if (2 * t.n + 1 < t.capacity) cudaEventRecord((cudaEvent_t)t.events[2 * t.n + 1], st);
    if (t.n < kTraceNames) t.names[t.n] = name;
    ++t.n;
}

namespace {

int fail(int code, const std::string& msg) {
    g_err = msg;
    return code;
}

int cuda_fail(int cerr, const char* what) {
    g_err = std::string(what) + ": " + cudaGetErrorName((cudaError_t)cerr) + " (" +
            cudaGetErrorString((cudaError_t)cerr) + ")";
    return MOE_ECUDA;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int check_shape(const moe_shape* s) {
    if (!s) return fail(MOE_EINVAL, "shape is NULL");
    if (s->T < 0) return fail(MOE_EINVAL, "T must be >= 0");
    if (s->H <= 0 || s->I <= 0) return fail(MOE_EINVAL, "H and I must be > 0");
    if (s->E < 1 || s->E > kMaxExperts) return fail(MOE_EINVAL, "E must be in [1, 1024]");
    static_assert(kMaxExperts == 1024, "update the E range in the message");
    if (s->k < 1 || s->k > s->E) return fail(MOE_EINVAL, "k must be in [1, E]");
    if (s->H % 64 || s->I % 64) return fail(MOE_EUNSUPPORTED, "H and I must be multiples of 64");
    if (s->block_m != kBM) return fail(MOE_EUNSUPPORTED, "block_m must be 128");
    if (!isfinite(s->activation_clamp)) return fail(MOE_EINVAL, "activation_clamp must be finite");
    if ((long long)s->T * s->k >= (1ll << 31)) return fail(MOE_EINVAL, "T*k must be < 2^31");
    const long long tk = (long long)s->T * s->k;
    const long long cap = tk + (long long)(tk < s->E ? tk : s->E) * (s->block_m - 1);
    if (cap * (long long)(2 * s->I) >= (1ll << 40) || cap >= (1ll << 31))
        return fail(MOE_EUNSUPPORTED, "routed rows exceed the supported range");
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- devices
int num_sms_current(int* out) {
    // filled on first use; host threads may race to fill it with the same value
    static std::atomic<int> cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached) {
        const int n = cache[dev].load(std::memory_order_relaxed);
        if (n > 0) {
            *out = n;
            return 0;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    if (cached) cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return 0;
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(std::string* err) {
    static EncodeTiledFn fn = nullptr;
    if (fn) return fn;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
        *err = "cuTensorMapEncodeTiled is not available from the driver";
        return nullptr;
    }
    fn = reinterpret_cast<EncodeTiledFn>(p);
    return fn;
}

// bf16 tensor map with 128-byte swizzle; dims innermost first, strides in
// bytes for dims 1..rank-1.
int make_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
             const cuuint32_t* box, const char* what, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B,
             CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    std::string err;
    EncodeTiledFn fn = encode_fn(&err);
    if (!fn) return fail(MOE_ECUDA, err);
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed for %s (CUresult %d)", what, (int)r);
        return fail(MOE_ECUDA, buf);
    }
    return MOE_OK;
}

// rows x cols bf16 matrix, box = box_cols x box_rows; a 64-byte-wide box uses
// the 64-byte swizzle, a 128-byte-wide box the 128-byte swizzle.
int map_2d(CUtensorMap* m, const void* p, long long rows, int cols, int box_cols, int box_rows, const char* what) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    return make_map(m, p, 2, dims, str, box, what,
                    box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
}

// [E][R][C] bf16, box = box_c x box_r x 1
int map_3d(CUtensorMap* m, const void* p, int E, int R, int C, int box_c, int box_r, const char* what) {
    cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)R, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)C * 2, (cuuint64_t)C * 2 * (cuuint64_t)R};
    cuuint32_t box[3] = {(cuuint32_t)box_c, (cuuint32_t)box_r, 1};
    return make_map(m, p, 3, dims, str, box, what);
}

// [E][R][C] f32 (a main gradient), box 32 x 32 x 1 (128-byte rows)
int map_3d_f32(CUtensorMap* m, const void* p, int E, int R, int C, const char* what) {
    cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)R, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)C * 4, (cuuint64_t)C * 4 * (cuuint64_t)R};
    cuuint32_t box[3] = {32, 32, 1};
    return make_map(m, p, 3, dims, str, box, what, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

// W1 [E][H][2I] viewed as [E][H][2][I] so that the gate and up halves are
// addressed separately and a tile never spills from one half into the other.
int map_w1_halves(CUtensorMap* m, const void* p, int E, int H, int I) {
    cuuint64_t dims[4] = {(cuuint64_t)I, 2, (cuuint64_t)H, (cuuint64_t)E};
    cuuint64_t str[3] = {(cuuint64_t)I * 2, (cuuint64_t)I * 4, (cuuint64_t)I * 4 * (cuuint64_t)H};
    cuuint32_t box[4] = {64, 1, 64, 1};
    return make_map(m, p, 4, dims, str, box, "W1 (gate/up halves)");
}

// E4M3 W1, K-major [E][2][I][H] bytes: a box is 128 bytes of K of 64 rows
// (columns) of one half, 128-byte swizzle.
int map_w1_fp8(CUtensorMap* m, const void* p, int E, int H, int I) {
    cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
    cuuint64_t str[3] = {(cuuint64_t)H, (cuuint64_t)H * I, (cuuint64_t)H * I * 2};
    cuuint32_t box[4] = {128, 64, 1, 1};
    return make_map(m, p, 4, dims, str, box, "W1 (E4M3, K-major)", CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// W1's scale atoms, E (I / 64) (H / 128) atoms of 512 bytes, as rows of 256
// bytes: a box is one atom (2 rows), no swizzle.
int map_w1_atoms(CUtensorMap* m, const void* p, int E, int H, int I) {
    cuuint64_t dims[2] = {256, (cuuint64_t)E * (I / 64) * (H / 128) * 2};
    cuuint64_t str[1] = {256};
    cuuint32_t box[2] = {256, 2};
    return make_map(m, p, 2, dims, str, box, "W1 scale atoms", CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// E4M3 W2, K-major [E][H][I] bytes: a box is 128 bytes of K of 128 rows,
// 128-byte swizzle.
int map_w2_fp8(CUtensorMap* m, const void* p, int E, int H, int I) {
    cuuint64_t dims[3] = {(cuuint64_t)I, (cuuint64_t)H, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)I, (cuuint64_t)I * H};
    cuuint32_t box[3] = {128, 128, 1};
    return make_map(m, p, 3, dims, str, box, "W2 (E4M3, K-major)", CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// W2's scale atoms, E (H / 128) (I / 128) atoms of 512 bytes, as rows of 256
// bytes: a box is one atom (2 rows), no swizzle.
int map_w2_atoms(CUtensorMap* m, const void* p, int E, int H, int I) {
    cuuint64_t dims[2] = {256, (cuuint64_t)E * (H / 128) * (I / 128) * 2};
    cuuint64_t str[1] = {256};
    cuuint32_t box[2] = {256, 2};
    return make_map(m, p, 2, dims, str, box, "W2 scale atoms", CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// E4M3 rows [rows][K] bytes: a box is 128 bytes of K of 32 rows, 128-byte
// swizzle.
int map_rows_fp8(CUtensorMap* m, const void* p, long long rows, int K, const char* what) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {128, 32};
    return make_map(m, p, 2, dims, str, box, what, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

struct Ctx {
    moe_layout L;
    int sms;
};

int prepare(const moe_shape* s, Ctx* c) {
    int rc = check_shape(s);
    if (rc) return rc;
    c->sms = 0;
    return compute_layout(s, &c->L);
}

// Called after every host-side argument check has passed.  Makes the device
// that owns `data` current on the calling thread (which may be a thread, such
// as an autograd worker, on which no CUDA context is current yet: tensor-map
// encoding needs one), then reads its SM count.
int query_device(Ctx* c, const void* data) {
    cudaPointerAttributes pa;
    cudaError_t e = cudaPointerGetAttributes(&pa, data);
    if (e != cudaSuccess) return cuda_fail((int)e, "querying the device of a workspace pointer");
    if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged)
        return fail(MOE_EINVAL, "workspace pointers must be device memory");
    e = cudaSetDevice(pa.device);
    if (e != cudaSuccess) return cuda_fail((int)e, "selecting the device");
    int r = num_sms_current(&c->sms);
    if (r) return cuda_fail(r, "querying the device");
    return MOE_OK;
}

GemmArgs base_args(const moe_shape* s, const moe_layout& L, uint8_t* route) {
    GemmArgs a;
    memset(&a, 0, sizeof a);
    a.T = s->T;
    a.H = s->H;
    a.I = s->I;
    a.E = s->E;
    a.k = s->k;
    a.tiles_cap = (int)L.tiles_cap;
    a.clamp = s->activation_clamp > 0.0f ? s->activation_clamp : INFINITY;
    a.dw_cols = L.dw_part_cols;
    a.perm = reinterpret_cast<const int32_t*>(route + L.perm);
    a.offs = reinterpret_cast<const int32_t*>(route + L.offs);
    a.counts = reinterpret_cast<const int32_t*>(route + L.counts);
    a.tiles = reinterpret_cast<const int32_t*>(route + L.tiles);
    a.pair_offs = reinterpret_cast<const int32_t*>(route + L.pair_offs);
    a.pair_owner = reinterpret_cast<const int32_t*>(route + L.pair_owner);
    a.status = reinterpret_cast<int32_t*>(route + L.status);
    return a;
}

int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace

int compute_layout(const moe_shape* s, moe_layout* L) {
    memset(L, 0, sizeof *L);
    const long long tk = (long long)s->T * s->k;
    const long long ne = tk < s->E ? tk : s->E;
    const long long bound = tk + ne * (s->block_m - 1);
    L->rows_cap = bound / s->block_m * s->block_m;
    L->tiles_cap = L->rows_cap / s->block_m;
    const size_t R = (size_t)L->rows_cap;
    const size_t A = 256;
    size_t o = 0;
    L->counts = o; o = align_up(o + 4 * (size_t)s->E, A);
    L->offs = o; o = align_up(o + 4 * (size_t)(s->E + 1), A);
    L->perm = o; o = align_up(o + 4 * R, A);
    L->inv = o; o = align_up(o + 4 * (size_t)tk, A);
    L->tiles = o; o = align_up(o + 4 * (size_t)L->tiles_cap, A);
    L->status = o; o = align_up(o + 4 * (size_t)MOE_STATUS_WORDS, A);
    L->pair_offs = o; o = align_up(o + 4 * (size_t)(s->E + 1), A);
    L->pair_owner = o; o = align_up(o + 4 * (size_t)L->tiles_cap, A);
    int nblk = 0;
    long long per_blk = 0;
    route_block_split(tk, &nblk, &per_blk);
    L->route_blocks = nblk;
    L->blk_counts = o; o = align_up(o + 4 * ((size_t)nblk * (size_t)(s->E + 1) + 1), A);
    L->route_bytes = o;
    o = 0;
    L->h = o; o = align_up(o + 2 * R * 2 * (size_t)s->I, A);
    L->a = o; o = align_up(o + 2 * R * (size_t)s->I, A);
    L->o = o; o = align_up(o + 2 * R * (size_t)s->H, A);
    L->cmask = o; o = align_up(o + 4 * R * (size_t)(2 * s->I / 32), A);
    L->saved_bytes = o;
    L->dw_part_cols = (s->I + 31) / 32;  // one partial per 32 features of the L2 dgrad epilogue
    o = 0;
    L->dh = o; o = align_up(o + 2 * R * 2 * (size_t)s->I, A);
    L->aw = o; o = align_up(o + 2 * R * (size_t)s->I, A);
    L->dxp = o; o = align_up(o + 2 * R * (size_t)s->H, A);
    L->dw_part = o; o = align_up(o + 4 * R * (size_t)L->dw_part_cols, A);
    L->bwd_bytes = o;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_workspace_layout(const moe_shape* shape, moe_layout* out) {
    if (!out) return fail(MOE_EINVAL, "out is NULL");
    int rc = check_shape(shape);
    if (rc) return rc;
    return compute_layout(shape, out);
}

int moe_route_prologue(const moe_shape* shape, const int32_t* topk_idx, void* route_ws, void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!route_ws || (shape->T > 0 && !topk_idx)) return fail(MOE_EINVAL, "NULL pointer argument");
    if (!aligned16(route_ws) || !aligned16(topk_idx)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if ((rc = query_device(&c, route_ws))) return rc;
    int e = launch_route_prologue(*shape, c.L, topk_idx, static_cast<uint8_t*>(route_ws), (cudaStream_t)stream);
    if (e) return cuda_fail(e, "route prologue launch");
    return MOE_OK;
}

int moe_router_topk(const moe_shape* shape, const float* logits, int32_t* topk_idx, float* topk_w, void* route_ws,
                    void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!route_ws || (shape->T > 0 && (!logits || !topk_idx || !topk_w))) return fail(MOE_EINVAL, "NULL pointer argument");
    const void* ptrs[] = {logits, topk_idx, topk_w, route_ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if ((rc = query_device(&c, route_ws))) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    trace_pre(st);
    int e = launch_router_topk(logits, shape->T, shape->E, shape->k, topk_idx, topk_w, c.sms, st);
    trace_post(st, "router_topk");
    if (e) return cuda_fail(e, "router top-k launch");
    e = launch_route_prologue(*shape, c.L, topk_idx, static_cast<uint8_t*>(route_ws), st);
    if (e) return cuda_fail(e, "route prologue launch");
    return MOE_OK;
}

// Body of moe_forward (x, W1, W2 bf16) and of moe_forward_fp8 (x8 / xsf the
// E4M3 input and its scales, W1 / w1sf and W2 / w2sf the E4M3 weights and
// their scale atoms).
static int forward_impl(const moe_shape* shape, const void* x, const uint8_t* x8, const uint8_t* xsf, const void* W1,
                        const uint8_t* w1sf, const void* W2, const uint8_t* w2sf, const float* topk_w, void* route_ws,
                        void* saved, void* y, void* stream, bool fp8) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!W1 || !W2 || !route_ws || !saved || (fp8 && (!w1sf || !w2sf)) ||
        (shape->T > 0 && (!topk_w || !y || (fp8 ? (!x8 || !xsf) : !x))))
        return fail(MOE_EINVAL, "NULL pointer argument");
    if (fp8 && (shape->H % 128 || shape->I % 128))
        return fail(MOE_EUNSUPPORTED, "the FP8 forward needs H and I to be multiples of 128");
    if (fp8 && shape->activation_clamp > 0.0f)
        return fail(MOE_EUNSUPPORTED, "the FP8 forward has no activation clamp");
    const void* ptrs[] = {x, x8, xsf, W1, w1sf, W2, w2sf, topk_w, route_ws, saved, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if ((rc = query_device(&c, route_ws))) return rc;
    if (shape->T == 0) return MOE_OK;
    const moe_layout& L = c.L;
    const int H = shape->H, I = shape->I, E = shape->E;
    uint8_t* route = static_cast<uint8_t*>(route_ws);
    uint8_t* sv = static_cast<uint8_t*>(saved);
    auto* h = reinterpret_cast<__nv_bfloat16*>(sv + L.h);
    auto* a = reinterpret_cast<__nv_bfloat16*>(sv + L.a);
    auto* o = reinterpret_cast<__nv_bfloat16*>(sv + L.o);
    auto* cmask = reinterpret_cast<uint32_t*>(sv + L.cmask);
    // FP8: a as E4M3 rows [rows_cap, I] and their scales [rows_cap, I / 32]
    // in a's region (which holds rows_cap I bf16)
    uint8_t* a8 = sv + L.a;
    uint8_t* asf = sv + L.a + (size_t)L.rows_cap * (size_t)I;
    cudaStream_t st = (cudaStream_t)stream;
    // L1 grouped GEMM (gathered x) + SwiGLU -> h, a; units of 128 gate and
    // 128 up features x one row chunk of one expert
    GemmMaps m1;
    memset(&m1, 0, sizeof m1);
    if (fp8) {
        if ((rc = map_w1_fp8(&m1.a, W1, E, H, I))) return rc;
        if ((rc = map_w1_atoms(&m1.b, w1sf, E, H, I))) return rc;
    } else if ((rc = map_w1_halves(&m1.a, W1, E, H, I))) {
        return rc;
    }
    if ((rc = map_2d(&m1.c0, h, L.rows_cap, 2 * I, 32, 32, "h (store)"))) return rc;
    if ((rc = map_2d(&m1.c1, a, L.rows_cap, I, 32, 32, "a (store)"))) return rc;
    GemmArgs g1 = base_args(shape, L, route);
    g1.K = H;
    g1.n_tiles = cdiv(I, 2 * 64);
    g1.gsrc = static_cast<const __nv_bfloat16*>(x);
    g1.gsrc8 = x8;
    g1.gsf = xsf;
    g1.cmask = cmask;
    if (fp8) {
        g1.q_out = a8;
        g1.sf_out = asf;
    }
    int e = launch_gemm(fp8 ? L1_FWD_MX : L1_FWD, g1, m1, (int)L.tiles_cap * g1.n_tiles, st);
    if (e) return cuda_fail(e, "L1 grouped GEMM launch");

    // L2 grouped GEMM + routing-weight epilogue -> o; units of 256 features
    GemmMaps m2;
    memset(&m2, 0, sizeof m2);
    if (fp8) {
        if ((rc = map_w2_fp8(&m2.a, W2, E, H, I))) return rc;
        if ((rc = map_rows_fp8(&m2.b, a8, L.rows_cap, I, "a (E4M3 rows)"))) return rc;
        if ((rc = map_w2_atoms(&m2.d, w2sf, E, H, I))) return rc;
    } else {
        if ((rc = map_3d(&m2.a, W2, E, I, H, 64, 64, "W2"))) return rc;
        if ((rc = map_2d(&m2.b, a, L.rows_cap, I, 64, 32, "a (rows)"))) return rc;
    }
    if ((rc = map_2d(&m2.c0, o, L.rows_cap, H, 32, 32, "o (store)"))) return rc;
    GemmArgs g2 = base_args(shape, L, route);
    g2.K = I;
    g2.n_tiles = cdiv(H, 2 * 128);
    g2.topk_w = topk_w;
    if (fp8) g2.gsf = asf;
    e = launch_gemm(fp8 ? L2_FWD_MX : L2_FWD, g2, m2, (int)L.tiles_cap * g2.n_tiles, st);
    if (e) return cuda_fail(e, "L2 grouped GEMM launch");

    // combine: y[t] = sum_j o[inv[t, j]]
    trace_pre(st);
    e = launch_combine(o, reinterpret_cast<const int32_t*>(route + L.inv), shape->T, shape->k, H,
                       static_cast<__nv_bfloat16*>(y), c.sms, st);
    trace_post(st, "combine_fwd");
    if (e) return cuda_fail(e, "combine launch");
    return MOE_OK;
}

int moe_forward(const moe_shape* shape, const void* x, const void* W1, const void* W2, const float* topk_w,
                void* route_ws, void* saved, void* y, void* stream) {
    return forward_impl(shape, x, nullptr, nullptr, W1, nullptr, W2, nullptr, topk_w, route_ws, saved, y, stream,
                        false);
}

int moe_forward_fp8(const moe_shape* shape, const uint8_t* x_fp8, const uint8_t* x_sf, const uint8_t* W1_fp8,
                    const uint8_t* W1_sf, const uint8_t* W2_fp8, const uint8_t* W2_sf, const float* topk_w,
                    void* route_ws, void* saved, void* y, void* stream) {
    return forward_impl(shape, nullptr, x_fp8, x_sf, W1_fp8, W1_sf, W2_fp8, W2_sf, topk_w, route_ws, saved, y, stream,
                        true);
}

int moe_quantize_weights_fp8(const moe_shape* shape, const void* W1, uint8_t* W1_fp8, uint8_t* W1_sf, void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!W1 || !W1_fp8 || !W1_sf) return fail(MOE_EINVAL, "NULL pointer argument");
    if (shape->H % 128) return fail(MOE_EUNSUPPORTED, "FP8 weights need H to be a multiple of 128");
    const void* ptrs[] = {W1, W1_fp8, W1_sf};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if ((rc = query_device(&c, W1))) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    trace_pre(st);
    const int e = launch_quantize_w1_fp8(static_cast<const __nv_bfloat16*>(W1), shape->E, shape->H, shape->I, W1_fp8,
                                         W1_sf, c.sms, st);
    trace_post(st, "quantize_w1_fp8");
    if (e) return cuda_fail(e, "W1 FP8 quantization launch");
    return MOE_OK;
}

int moe_quantize_w2_fp8(const moe_shape* shape, const void* W2, uint8_t* W2_fp8, uint8_t* W2_sf, void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!W2 || !W2_fp8 || !W2_sf) return fail(MOE_EINVAL, "NULL pointer argument");
    if (shape->H % 128 || shape->I % 128)
        return fail(MOE_EUNSUPPORTED, "FP8 W2 needs H and I to be multiples of 128");
    const void* ptrs[] = {W2, W2_fp8, W2_sf};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if ((rc = query_device(&c, W2))) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    trace_pre(st);
    const int e = launch_quantize_w2_fp8(static_cast<const __nv_bfloat16*>(W2), shape->E, shape->H, shape->I, W2_fp8,
                                         W2_sf, c.sms, st);
    trace_post(st, "quantize_w2_fp8");
    if (e) return cuda_fail(e, "W2 FP8 quantization launch");
    return MOE_OK;
}

int moe_dequantize_fp8(const moe_shape* shape, const uint8_t* x_fp8, const uint8_t* x_sf, void* x_out, void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (shape->T > 0 && (!x_fp8 || !x_sf || !x_out)) return fail(MOE_EINVAL, "NULL pointer argument");
    const void* ptrs[] = {x_fp8, x_sf, x_out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if (shape->T == 0) return MOE_OK;
    if ((rc = query_device(&c, x_out))) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    trace_pre(st);
    const int e = launch_dequantize_fp8(x_fp8, x_sf, (long long)shape->T * shape->H,
                                        static_cast<__nv_bfloat16*>(x_out), c.sms, st);
    trace_post(st, "dequantize_fp8");
    if (e) return cuda_fail(e, "FP8 dequantization launch");
    return MOE_OK;
}

int moe_quantize_fp8(const moe_shape* shape, const void* x, uint8_t* x_fp8, uint8_t* x_sf, void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (shape->T > 0 && (!x || !x_fp8 || !x_sf)) return fail(MOE_EINVAL, "NULL pointer argument");
    const void* ptrs[] = {x, x_fp8, x_sf};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if (shape->T == 0) return MOE_OK;
    if ((rc = query_device(&c, x))) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    trace_pre(st);
    const int e = launch_quantize_fp8(static_cast<const __nv_bfloat16*>(x), (long long)shape->T * shape->H, x_fp8,
                                      x_sf, c.sms, st);
    trace_post(st, "quantize_fp8");
    if (e) return cuda_fail(e, "FP8 quantization launch");
    return MOE_OK;
}

// Body of moe_backward (main_grad false: dW1/dW2 bf16, overwritten) and of
// moe_backward_main_grad (main_grad true: dW1/dW2 are the FP32 main
// gradients, added to).
static int backward_impl(const moe_shape* shape, const void* dY, const void* x, const void* W1, const void* W2,
                  const float* topk_w, void* route_ws, const void* saved, void* bwd_ws, void* dx, void* dW1, void* dW2,
                  float* dtopk_w, void* stream, bool main_grad) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!W1 || !W2 || !route_ws || !saved || !bwd_ws || !dW1 || !dW2 ||
        (shape->T > 0 && (!dY || !x || !topk_w || !dx || !dtopk_w)))
        return fail(MOE_EINVAL, "NULL pointer argument");
    const void* ptrs[] = {dY, x, W1, W2, topk_w, route_ws, saved, bwd_ws, dx, dW1, dW2, dtopk_w};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    if ((rc = query_device(&c, route_ws))) return rc;
    const moe_layout& L = c.L;
    const int H = shape->H, I = shape->I, E = shape->E;
    cudaStream_t st = (cudaStream_t)stream;
    if (shape->T == 0) {
        if (main_grad) return MOE_OK;  // nothing to add
        cudaError_t ce = cudaMemsetAsync(dW1, 0, (size_t)E * H * 2 * I * 2, st);
        if (ce == cudaSuccess) ce = cudaMemsetAsync(dW2, 0, (size_t)E * I * H * 2, st);
        if (ce != cudaSuccess) return cuda_fail((int)ce, "zeroing weight gradients");
        return MOE_OK;
    }
    uint8_t* route = static_cast<uint8_t*>(route_ws);
    const uint8_t* sv = static_cast<const uint8_t*>(saved);
    uint8_t* ws = static_cast<uint8_t*>(bwd_ws);
    auto* h = reinterpret_cast<const __nv_bfloat16*>(sv + L.h);
    auto* a = reinterpret_cast<const __nv_bfloat16*>(sv + L.a);
    auto* dh = reinterpret_cast<__nv_bfloat16*>(ws + L.dh);
    auto* aw = reinterpret_cast<__nv_bfloat16*>(ws + L.aw);
    auto* dxp = reinterpret_cast<__nv_bfloat16*>(ws + L.dxp);
    auto* dwp = reinterpret_cast<float*>(ws + L.dw_part);
    const auto* inv = reinterpret_cast<const int32_t*>(route + L.inv);
    // L2 dgrad (gathered dY) + SwiGLU^T -> dh, aw, dw_part; units of 256
    // features of I
    GemmMaps m;
    memset(&m, 0, sizeof m);
    if ((rc = map_3d(&m.a, W2, E, I, H, 64, 128, "W2 (K-major)"))) return rc;
    if ((rc = map_2d(&m.b, h, L.rows_cap, 2 * I, 32, 32, "h (epilogue input)"))) return rc;
    if ((rc = map_2d(&m.d, a, L.rows_cap, I, 32, 32, "a (epilogue input)"))) return rc;
    if ((rc = map_2d(&m.c0, dh, L.rows_cap, 2 * I, 32, 32, "dh (store)"))) return rc;
    if ((rc = map_2d(&m.c1, aw, L.rows_cap, I, 32, 32, "aw (store)"))) return rc;
    GemmArgs g = base_args(shape, L, route);
    g.K = H;
    g.n_tiles = cdiv(I, 2 * 128);
    g.gsrc = static_cast<const __nv_bfloat16*>(dY);
    g.topk_w = topk_w;
    g.h_in = h;
    g.a_in = a;
    g.cmask = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(sv + L.cmask));
    g.outf = dwp;
    int e = launch_gemm(L2_DGRAD, g, m, (int)L.tiles_cap * g.n_tiles, st);
    if (e) return cuda_fail(e, "L2 dgrad launch");

    // dW2[e] = aw_e^T . dY_e (variable K)
    GemmMaps m3;
    memset(&m3, 0, sizeof m3);
    if ((rc = map_2d(&m3.a, aw, L.rows_cap, I, 64, 64, "aw"))) return rc;
    if ((rc = main_grad ? map_3d_f32(&m3.c0, dW2, E, I, H, "main_grad_W2 (reduce-add)")
                        : map_3d(&m3.c0, dW2, E, I, H, 64, 32, "dW2 (store)")))
        return rc;
    // units: (expert, 256 features of H); each streams the expert's aw in
    // tiles of 256 features of I
    GemmArgs g3 = base_args(shape, L, route);
    g3.m_tiles = cdiv(H, 256);
    g3.n_tiles = cdiv(I, 256);
    g3.gsrc = static_cast<const __nv_bfloat16*>(dY);
    e = launch_gemm(main_grad ? DW2_MG : DW2, g3, m3, E * g3.m_tiles, st);
    if (e) return cuda_fail(e, "dW2 launch");

    // dW1[e] = x_e^T . dh_e (variable K, x re-gathered)
    GemmMaps m4;
    memset(&m4, 0, sizeof m4);
    if ((rc = map_2d(&m4.b, dh, L.rows_cap, 2 * I, 64, 64, "dh (rows)"))) return rc;
    if ((rc = main_grad ? map_3d_f32(&m4.c0, dW1, E, H, 2 * I, "main_grad_W1 (reduce-add)")
                        : map_3d(&m4.c0, dW1, E, H, 2 * I, 64, 32, "dW1 (store)")))
        return rc;
    // units: (expert, 256 features of H); each streams the expert's dh in
    // tiles of 256 features of 2I
    GemmArgs g4 = base_args(shape, L, route);
    g4.m_tiles = cdiv(H, 256);
    g4.n_tiles = cdiv(2 * I, 256);
    g4.gsrc = static_cast<const __nv_bfloat16*>(x);
    e = launch_gemm(main_grad ? DW1_MG : DW1, g4, m4, E * g4.m_tiles, st);
    if (e) return cuda_fail(e, "dW1 launch");

    // L1 dgrad: dxp = dh . W1[e]^T; units of 256 features of H
    GemmMaps m5;
    memset(&m5, 0, sizeof m5);
    if ((rc = map_3d(&m5.a, W1, E, H, 2 * I, 64, 128, "W1 (K-major)"))) return rc;
    if ((rc = map_2d(&m5.b, dh, L.rows_cap, 2 * I, 64, 32, "dh (rows)"))) return rc;
    if ((rc = map_2d(&m5.c0, dxp, L.rows_cap, H, 32, 32, "dxp (store)"))) return rc;
    GemmArgs g5 = base_args(shape, L, route);
    g5.K = 2 * I;
    g5.n_tiles = cdiv(H, 2 * 128);
    e = launch_gemm(L1_DGRAD, g5, m5, (int)L.tiles_cap * g5.n_tiles, st);
    if (e) return cuda_fail(e, "L1 dgrad launch");

    // backward combine and the routing-weight gradient
    trace_pre(st);
    e = launch_combine(dxp, inv, shape->T, shape->k, H, static_cast<__nv_bfloat16*>(dx), c.sms, st);
    trace_post(st, "combine_bwd");
    if (e) return cuda_fail(e, "backward combine launch");
    trace_pre(st);
    e = launch_dw_reduce(dwp, L.dw_part_cols, inv, (long long)shape->T * shape->k, dtopk_w, c.sms, st);
    trace_post(st, "dw_reduce");
    if (e) return cuda_fail(e, "d(topk_weights) reduce launch");
    return MOE_OK;
}

int moe_backward(const moe_shape* shape, const void* dY, const void* x, const void* W1, const void* W2,
                 const float* topk_w, void* route_ws, const void* saved, void* bwd_ws, void* dx, void* dW1,
                 void* dW2, float* dtopk_w, void* stream) {
    return backward_impl(shape, dY, x, W1, W2, topk_w, route_ws, saved, bwd_ws, dx, dW1, dW2, dtopk_w, stream,
                         false);
}

int moe_backward_main_grad(const moe_shape* shape, const void* dY, const void* x, const void* W1, const void* W2,
                           const float* topk_w, void* route_ws, const void* saved, void* bwd_ws, void* dx,
                           float* main_grad_W1, float* main_grad_W2, float* dtopk_w, void* stream) {
    return backward_impl(shape, dY, x, W1, W2, topk_w, route_ws, saved, bwd_ws, dx, main_grad_W1, main_grad_W2,
                         dtopk_w, stream, true);
}

int moe_read_status(const moe_shape* shape, const void* route_ws, int32_t* out, void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!route_ws || !out) return fail(MOE_EINVAL, "NULL pointer argument");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(out, static_cast<const uint8_t*>(route_ws) + c.L.status,
                                    sizeof(int32_t) * MOE_STATUS_WORDS, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail((int)e, "reading status words");
    return MOE_OK;
}

int moe_selftest_wait_timeout(const moe_shape* shape, void* route_ws, uint64_t limit_ns, int64_t* elapsed_ns,
                              void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!route_ws) return fail(MOE_EINVAL, "NULL pointer argument");
    if (!aligned16(route_ws) || (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u))
        return fail(MOE_EUNSUPPORTED, "route_ws must be 16-byte and elapsed_ns 8-byte aligned");
    if (limit_ns < 1000u || limit_ns > 100000000u)
        return fail(MOE_EINVAL, "limit_ns must be in [1 us, 100 ms]");
    if ((rc = query_device(&c, route_ws))) return rc;
    int32_t* status = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(route_ws) + c.L.status);
    const int e = launch_wait_selftest(status, limit_ns, reinterpret_cast<long long*>(elapsed_ns),
                                       (cudaStream_t)stream);
    if (e) return cuda_fail(e, "bounded-wait self-test launch");
    return MOE_OK;
}

int moe_trace_begin(void* const* events, int capacity) {
    if (capacity < 0 || (capacity > 0 && !events)) return fail(MOE_EINVAL, "bad trace event array");
    g_trace.events = capacity > 0 ? events : nullptr;
    g_trace.capacity = capacity;
    g_trace.n = 0;
    return MOE_OK;
}

int moe_trace_end(void) {
    const int n = g_trace.n;
    g_trace.events = nullptr;
    g_trace.capacity = 0;
    return n;
}

const char* moe_trace_kernel(int i) {
    if (i < 0 || i >= g_trace.n || i >= kTraceNames) return "";
    return g_trace.names[i];
}

const char* moe_last_error(void) { return g_err.c_str(); }

const char* moe_version(void) { return "moe_gb300 0.1 (sm_103a, tcgen05)"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Inference forward for callers that cannot allocate device memory.
//
// The routing tables and the per-row intermediates (h, a, o) live in one
// file-scope device array instead of caller workspaces.  Every GPU that loads
// this library holds the array (kNoAllocScratchBytes) until the process exits.
// Host code cannot use the array's name as a device address, so the address is
// fetched once per device with cudaGetSymbolAddress, with that device current.
namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set-up on the
// first call per device).  The address is kept for the life of the process:
// after a cudaDeviceReset of that device it would be stale, so the entry
// point is not for use across a device reset.
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail((int)e, "querying the current device");
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_EUNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return cuda_fail((int)(e != cudaSuccess ? e : cudaErrorInvalidSymbol),
                                                     "cudaGetSymbolAddress of the static scratch");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_forward_noalloc(const moe_shape* shape, const void* x, const void* W1, const void* W2,
                                   const int32_t* topk_idx, const float* topk_w, void* y, int32_t* status_out,
                                   void* stream) {
    Ctx c;
    int rc = prepare(shape, &c);
    if (rc) return rc;
    if (!W1 || !W2 || (shape->T > 0 && (!x || !topk_idx || !topk_w || !y)))
        return fail(MOE_EINVAL, "NULL pointer argument");
    const void* ptrs[] = {x, W1, W2, topk_idx, topk_w, y, status_out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MOE_EUNSUPPORTED, "pointers must be 16-byte aligned");
    const size_t route_part = align_up(c.L.route_bytes, 256);
    const size_t need = route_part + c.L.saved_bytes;
    if (need > kNoAllocScratchBytes) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "moe_forward_noalloc: this shape needs %zu bytes of scratch, more than the %zu-byte static "
                 "scratch; use moe_forward with caller workspaces",
                 need, kNoAllocScratchBytes);
        return fail(MOE_EUNSUPPORTED, buf);
    }
    if ((rc = query_device(&c, W1))) return rc;
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch))) return rc;
    uint8_t* route = static_cast<uint8_t*>(scratch);
    // The prologue rewrites every table and status word it owns on each call,
    // so nothing left by an earlier call is read.
    if ((rc = moe_route_prologue(shape, topk_idx, route, stream))) return rc;
    if ((rc = moe_forward(shape, x, W1, W2, topk_w, route, route + route_part, y, stream))) return rc;
    if (status_out) {
        // the status words stay in the static scratch, which the caller
        // cannot address: copy them out (device to device, on the stream)
        const cudaError_t e = cudaMemcpyAsync(status_out, route + c.L.status, sizeof(int32_t) * MOE_STATUS_WORDS,
                                              cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail((int)e, "copying the status words out of the static scratch");
    }
    return MOE_OK;
}
