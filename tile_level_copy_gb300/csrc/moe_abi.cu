// Host side of libmoe: argument checks, workspace layout, TMA descriptors and the launch
// sequences behind the C ABI declared in include/moe.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "moe_internal.cuh"

namespace moe {
namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    moe_layout L;
    Shape S;
};

// Checks the config and derives the workspace layout and the kernel shape.
int make_layout(const moe_config* c, Layout* out) {
    if (!c) return fail(MOE_ERR_ARG, "config is NULL");
    const int64_t T = c->T, d = c->d, F = c->ffn, E = c->E, k = c->topk, R = c->R, tbM = c->tile_M;
    if (T <= 0 || d <= 0 || F <= 0 || E <= 0 || k <= 0 || R <= 0)
        return fail(MOE_ERR_ARG, "T, d, ffn, E, topk, R must be positive");
    if (d % 128) return fail(MOE_ERR_ARG, "d=%lld must be a multiple of 128", (long long)d);
    if (F % 128) return fail(MOE_ERR_ARG, "ffn=%lld must be a multiple of 128", (long long)F);
    if (E > MAX_E) return fail(MOE_ERR_ARG, "E=%lld exceeds %d", (long long)E, MAX_E);
    if (k > E || k > 8) return fail(MOE_ERR_ARG, "topk=%lld must be <= min(E, 8)", (long long)k);
    if (T % R) return fail(MOE_ERR_ARG, "R=%lld must divide T=%lld", (long long)R, (long long)T);
    if (E * R > 1024) return fail(MOE_ERR_ARG, "E*R=%lld exceeds 1024", (long long)(E * R));
    if (tbM != 64 && tbM != 128) return fail(MOE_ERR_ARG, "tile_M=%lld must be 64 or 128", (long long)tbM);
    if (c->mgb < 1 || c->mgb > 4) return fail(MOE_ERR_ARG, "mgb=%d must be in [1, 4]", c->mgb);
    for (int i = 0; i < 4; ++i)
        if (c->reserved[i]) return fail(MOE_ERR_ARG, "reserved fields must be zero");
    if (c->tail_window < 0) return fail(MOE_ERR_ARG, "tail_window=%d must be >= 0", c->tail_window);

    const int64_t TK = T * k, G = E * R;
    const int64_t P_max = (int64_t)align_up((size_t)(TK + (G < TK ? G : TK) * (tbM - 1)), (size_t)tbM);
    if (P_max >= (int64_t(1) << 30)) return fail(MOE_ERR_ARG, "padded rows %lld too large", (long long)P_max);
    const int64_t MT_max = P_max / tbM;
    const int64_t PC_max = (int64_t)align_up((size_t)(TK + (E < TK ? E : TK) * (BM - 1)), (size_t)BM);
    const int64_t IU_max = PC_max / BM;
    // route chunk: <= 128 tokens and <= 32 KB of staged logits, a power of two dividing T/R
    int64_t C = 128;
    while (C > 1 && C * (E + 1) * 4 > 32768) C >>= 1;
    while ((T / R) % C) C >>= 1;
    const int bn2 = (d % 256 == 0) ? 256 : 128;
    const int nN2 = (int)(d / bn2);
    if ((int64_t)c->mgb * nN2 > GEMM_THREADS)
        return fail(MOE_ERR_ARG, "mgb * d/%d = %lld exceeds %d", bn2, (long long)c->mgb * nN2, GEMM_THREADS);
    auto rows_for = [&](int64_t bytes) {
        int64_t r = bytes / (2 * d);
        return r < 1 ? int64_t(1) : (r > tbM ? tbM : r);
    };
    const int64_t rpu = rows_for(UNIT_BYTES), rpu_tail = rows_for(TAIL_UNIT_BYTES);

    Layout o;
    memset(&o, 0, sizeof(o));
    moe_layout& L = o.L;
    L.P_max = (int32_t)P_max;
    L.MT_max = (int32_t)MT_max;
    L.PC_max = (int32_t)PC_max;
    L.IU_max = (int32_t)IU_max;
    L.n_chunks = (int32_t)(T / C);
    L.chunk_tokens = (int32_t)C;
    L.n_tiles_n2 = nN2;
    L.block_n2 = bn2;
    L.rows_per_unit = (int32_t)rpu;
    L.units_per_band = (int32_t)((tbM + rpu - 1) / rpu);

    size_t cur = 0;
    auto put = [&](size_t bytes) {
        const size_t at = cur;
        cur = align_up(cur + bytes, 1024);
        return at;
    };
    L.idx = put(TK * 4);
    L.gate = put(TK * 4);
    L.rank = put(TK * 4);
    L.chunk_cnt = put((size_t)L.n_chunks * E * 4);
    L.chunk_base = put((size_t)L.n_chunks * E * 4);
    L.counts = put(G * 4);
    L.offsets = put((G + 1) * 4);
    L.ret_off = put(R * (E + 1) * 4);
    L.tiles = put(MT_max * 16);
    L.tile_ret = put(MT_max * 4);
    L.sched = put(MT_max * 4);
    L.order = put(MT_max * 4);
    L.seg = put(MT_max * 8);
    L.experts = put(E * 32);
    L.items_up = put(IU_max * 8);
    L.items_down = put(MT_max * 8);
    L.slot = put(TK * 4);
    L.cslot = put(TK * 4);
    L.ret_slot = put(TK * 4);
    L.yrow = put(PC_max * 4);
    L.tile_crow = put(MT_max * 4);
    L.band_item = put(MT_max * 4);
    L.tok_of = put(PC_max * 4);
    L.xrows = put(E * 4);
    L.xready = put(E * 4);
    L.meta = put(META_COUNT * 4);
    L.flags = put(MT_max * nN2 * 4);
    L.bands = put(MT_max * 4);
    L.trace = put(TR_COUNT * 8);
    L.Xc = put((size_t)PC_max * d * 2);
    L.Hc = put((size_t)PC_max * F * 2);
    L.Yp = put((size_t)P_max * d * 2);
    L.Ret = put((size_t)TK * d * 2);
    L.in_logits = put(2 * (size_t)T * E * 4);
    L.in_x = put(2 * (size_t)T * d * 2);
    L.out = put(2 * (size_t)T * d * 4);
    L.bytes = cur;

    Shape& S = o.S;
    S.T = (int)T;
    S.d = (int)d;
    S.ffn = (int)F;
    S.E = (int)E;
    S.k = (int)k;
    S.R = (int)R;
    S.tbM = (int)tbM;
    S.mgb = c->mgb;
    S.chunk_tokens = (int)C;
    S.n_chunks = L.n_chunks;
    S.P_max = L.P_max;
    S.MT_max = L.MT_max;
    S.PC_max = L.PC_max;
    S.IU_max = L.IU_max;
    S.bn2 = bn2;
    S.n_tiles_n2 = nN2;
    S.rows_per_unit = L.rows_per_unit;
    S.units_per_band = L.units_per_band;
    S.rows_per_unit_tail = (int)rpu_tail;
    S.units_per_band_tail = (int)((tbM + rpu_tail - 1) / rpu_tail);
    S.tail_bands = (TAIL_TILES + nN2 - 1) / nN2;
    // An expert's W2 of at least half the L2 (128 MB) is streamed from DRAM again by each wave its
    // band-first tiles span; N tile by N tile, each W2 tile is read by pair items that run together,
    // but each item's rows are read once per N tile, so that order is taken only by experts whose
    // rows (items x 128 x ffn x 2 bytes) fit in half the L2 as well. Smaller W2 stay in L2 across
    // waves, and there band-first order keeps each item's rows hot.
    const int64_t half_l2 = int64_t(64) << 20;
    S.down_n_outer_items = (d * F * 2 >= half_l2) ? (int)(half_l2 / (int64_t(BM) * F * 2)) : 0;
    S.timeout_ns = (unsigned long long)(c->timeout_us ? c->timeout_us : 2000000u) * 1000ull;
    S.flags = c->flags;
    S.tail_window = c->tail_window;
    *out = o;
    return MOE_OK;
}

PlanPtrs plan_ptrs(const moe_layout& L, void* ws) {
    uint8_t* b = static_cast<uint8_t*>(ws);
    PlanPtrs p{};  // host_rec stays null except in moe_forward_dma
    p.idx = reinterpret_cast<int32_t*>(b + L.idx);
    p.gate = reinterpret_cast<float*>(b + L.gate);
    p.rank = reinterpret_cast<int32_t*>(b + L.rank);
    p.chunk_cnt = reinterpret_cast<int32_t*>(b + L.chunk_cnt);
    p.chunk_base = reinterpret_cast<int32_t*>(b + L.chunk_base);
    p.counts = reinterpret_cast<int32_t*>(b + L.counts);
    p.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
    p.ret_off = reinterpret_cast<int32_t*>(b + L.ret_off);
    p.tiles = reinterpret_cast<int32_t*>(b + L.tiles);
    p.tile_ret = reinterpret_cast<int32_t*>(b + L.tile_ret);
    p.sched = reinterpret_cast<int32_t*>(b + L.sched);
    p.order = reinterpret_cast<int32_t*>(b + L.order);
    p.seg = reinterpret_cast<int32_t*>(b + L.seg);
    p.experts = reinterpret_cast<int32_t*>(b + L.experts);
    p.items_up = reinterpret_cast<int32_t*>(b + L.items_up);
    p.items_down = reinterpret_cast<int32_t*>(b + L.items_down);
    p.slot = reinterpret_cast<int32_t*>(b + L.slot);
    p.cslot = reinterpret_cast<int32_t*>(b + L.cslot);
    p.ret_slot = reinterpret_cast<int32_t*>(b + L.ret_slot);
    p.yrow = reinterpret_cast<int32_t*>(b + L.yrow);
    p.tile_crow = reinterpret_cast<int32_t*>(b + L.tile_crow);
    p.band_item = reinterpret_cast<int32_t*>(b + L.band_item);
    p.tok_of = reinterpret_cast<int32_t*>(b + L.tok_of);
    p.xrows = reinterpret_cast<uint32_t*>(b + L.xrows);
    p.xready = reinterpret_cast<uint32_t*>(b + L.xready);
    p.meta = reinterpret_cast<int32_t*>(b + L.meta);
    p.flags = reinterpret_cast<uint32_t*>(b + L.flags);
    p.bands = reinterpret_cast<uint32_t*>(b + L.bands);
    p.trace = reinterpret_cast<unsigned long long*>(b + L.trace);
    p.Xc = reinterpret_cast<__nv_bfloat16*>(b + L.Xc);
    p.Hc = reinterpret_cast<__nv_bfloat16*>(b + L.Hc);
    p.Yp = reinterpret_cast<__nv_bfloat16*>(b + L.Yp);
    p.Ret = reinterpret_cast<__nv_bfloat16*>(b + L.Ret);
    return p;
}

// ---- device query ------------------------------------------------------------------------------
struct DeviceInfo {
    int sms = 0;
    bool supported = false;
};

int device_info(DeviceInfo* di) {
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    di->sms = sms;
    di->supported = (major == 10 && minor == 3);
    return MOE_OK;
}

// ---- TMA descriptors ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 tensor [outer][mid][inner] (rank 3) or [mid][inner] (rank 2, outer = 1); box box_inner x
// box_mid (x 1). Operand maps: 64-element inner box with the 128-byte swizzle the UMMA descriptors
// expect; output maps: 32 x 32 boxes, unswizzled (row pitch 64 bytes in shared memory).
// Out-of-bounds elements read as zero.
int make_map(CUtensorMap* m, const void* ptr, int rank, uint64_t inner, uint64_t mid, uint64_t outer,
             uint32_t box_mid, const char* what, uint32_t box_inner = BK, bool swizzle = true) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {inner, mid, outer};
    cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
    cuuint32_t box[3] = {box_inner, box_mid, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
    return MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Call {
    Layout lay;
    PlanPtrs p;
    DeviceInfo di;
    cudaStream_t st;
    int consumers;
};

int begin_call(const moe_config* cfg, void* ws, size_t ws_bytes, void* stream, Call* c) {
    g_err.clear();
    int rc = make_layout(cfg, &c->lay);
    if (rc) return rc;
    if (!ws) return fail(MOE_ERR_ARG, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_ARG, "workspace must be 256-byte aligned");
    if (ws_bytes < c->lay.L.bytes)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, c->lay.L.bytes);
    rc = device_info(&c->di);
    if (rc) return rc;
    if (!c->di.supported) return fail(MOE_ERR_DEVICE, "current device is not sm_103 (GB300)");
    c->p = plan_ptrs(c->lay.L, ws);
    c->st = static_cast<cudaStream_t>(stream);
    c->consumers = cfg->consumer_ctas;
    return MOE_OK;
}

int run_plan(Call& c, const float* logits, const uint16_t* x, bool permute) {
    cudaError_t e = launch_route(c.lay.S, logits, c.p, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "route kernel launch");
    e = launch_plan(c.lay.S, c.p, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "plan kernel launch");
    e = launch_permute(c.lay.S, permute ? reinterpret_cast<const __nv_bfloat16*>(x) : nullptr, c.p, c.di.sms, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "permute kernel launch");
    return MOE_OK;
}

// Records a caller's stage event. While `st` is being captured into a CUDA graph the record becomes
// an event-record node of the graph (cudaEventRecordExternal), so every replay records it: timing a
// graph of several steps then gives each kernel's duration inside the replayed region.
int record(void* const* ev, int i, cudaStream_t st) {
    if (!ev || !ev[i]) return MOE_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e == cudaSuccess)
        e = (cs == cudaStreamCaptureStatusActive)
                ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev[i]), st, cudaEventRecordExternal)
                : cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "cudaEventRecord of a stage event");
}

int run_forward(Call& c, const float* logits, const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                const uint16_t* W2, float* out, bool overlapped, void* const* ev = nullptr) {
    const Shape& S = c.lay.S;
    const moe_layout& L = c.lay.L;
    if (!logits || !x || !W1 || !W3 || !W2 || !out) return fail(MOE_ERR_ARG, "NULL input or output pointer");
    if (!aligned(x, 16) || !aligned(W1, 16) || !aligned(W3, 16) || !aligned(W2, 16) || !aligned(out, 16) ||
        !aligned(logits, 4))
        return fail(MOE_ERR_ARG, "x, W1, W3, W2, out must be 16-byte aligned, logits 4-byte aligned");
    const int min_consumers = (S.flags & MOE_COPY_WARPS) ? 0 : 1;
    if (overlapped && (c.consumers < min_consumers || c.consumers > c.di.sms / 2))
        return fail(MOE_ERR_ARG, "consumer_ctas=%d must be in [%d, %d]", c.consumers, min_consumers, c.di.sms / 2);

    // The down-projection runs on CTA pairs with MOE_PAIR_UMMA when its UMMA tile is 256 columns wide,
    // the consumer partition is whole clusters and no copy warps are asked for; the sequential
    // baseline of the same configuration uses the same kernel.
    const bool pair_down = (S.flags & MOE_PAIR_UMMA) && !(S.flags & MOE_COPY_WARPS) && S.bn2 == 2 * BN1 &&
                           (c.consumers % 2 == 0);
    CUtensorMap tXc, tHc, tW1, tW3, tW2, tW2h, tHcOut, tYpOut;
    int rc = make_map(&tXc, c.p.Xc, 2, S.d, S.PC_max, 1, BM, "Xc");
    if (!rc) rc = make_map(&tHc, c.p.Hc, 2, S.ffn, S.PC_max, 1, BM, "Hc");
    if (!rc) rc = make_map(&tHcOut, c.p.Hc, 2, S.ffn, S.PC_max, 1, 32, "Hc (store)", EPI_CHUNK, false);
    if (!rc) rc = make_map(&tYpOut, c.p.Yp, 2, S.d, S.P_max, 1, 32, "Yp (store)", EPI_CHUNK, false);
    if (!rc) rc = make_map(&tW1, W1, 3, S.d, S.ffn, S.E, BN1, "W1");
    if (!rc) rc = make_map(&tW3, W3, 3, S.d, S.ffn, S.E, BN1, "W3");
    if (!rc) rc = make_map(&tW2, W2, 3, S.ffn, S.d, S.E, S.bn2, "W2");
    if (!rc && pair_down) rc = make_map(&tW2h, W2, 3, S.ffn, S.d, S.E, BN1, "W2 (half)");
    if (rc) return rc;
    (void)L;

    if ((rc = record(ev, MOE_EV_BEGIN, c.st))) return rc;
    // with MOE_FUSED_DISPATCH the permute only computes the slots; the SwiGLU GEMM copies the rows
    const bool fused_dispatch = (S.flags & MOE_FUSED_DISPATCH) != 0;
    c.p.x = reinterpret_cast<const __nv_bfloat16*>(x);
    rc = run_plan(c, logits, x, !fused_dispatch);
    if (rc) return rc;
    if ((rc = record(ev, MOE_EV_PLANNED, c.st))) return rc;
    cudaError_t e;
    if (overlapped && pair_down && (S.flags & MOE_FUSED_GEMMS)) {
        // both GEMMs in one launch: the stage events after it mark the end of both
        e = launch_gemm_fused_pair(S, c.p, tXc, tW1, tW3, tHcOut, tHc, tW2h, tYpOut, c.consumers, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "fused GEMM launch");
        if ((rc = record(ev, MOE_EV_UP, c.st))) return rc;
        if ((rc = record(ev, MOE_EV_DOWN, c.st))) return rc;
        if ((rc = record(ev, MOE_EV_COPIED, c.st))) return rc;
        e = launch_combine(S, c.p, out, c.di.sms, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
        return record(ev, MOE_EV_END, c.st);
    }
    e = (S.flags & MOE_PAIR_UMMA) ? launch_gemm_swiglu_pair(S, c.p, tXc, tW1, tW3, tHcOut, c.st)
                                  : launch_gemm_swiglu(S, c.p, tXc, tW1, tW3, tHcOut, c.di.sms, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "SwiGLU GEMM launch");
    if ((rc = record(ev, MOE_EV_UP, c.st))) return rc;
    if (overlapped) {
        e = pair_down ? launch_gemm_down_pair(S, c.p, tHc, tW2h, tYpOut, c.consumers, true, c.st)
                      : launch_gemm_down(S, c.p, tHc, tW2, tYpOut, c.di.sms, c.consumers, true, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "overlapped down-projection launch");
        if ((rc = record(ev, MOE_EV_DOWN, c.st))) return rc;
    } else {
        e = pair_down ? launch_gemm_down_pair(S, c.p, tHc, tW2h, tYpOut, 0, false, c.st)
                      : launch_gemm_down(S, c.p, tHc, tW2, tYpOut, c.di.sms, 0, false, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "down-projection launch");
        if ((rc = record(ev, MOE_EV_DOWN, c.st))) return rc;
        e = launch_copy_seq(S, c.p, c.di.sms, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "return copy launch");
    }
    if ((rc = record(ev, MOE_EV_COPIED, c.st))) return rc;
    e = launch_combine(S, c.p, out, c.di.sms, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return record(ev, MOE_EV_END, c.st);
}

}  // namespace
}  // namespace moe

// ---- static-scratch routing plan ------------------------------------------------------------------
// Scratch of moe_route_static: one file-scope array per GPU that loads the library, kept until the
// process exits. Host code must not pass `g_static_scratch` itself to a kernel (on the host the name
// is only a stand-in); the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

namespace moe {
namespace {

// Offsets of the plan's scratch regions inside the static array for one config (256-byte aligned).
struct StaticLayout {
    size_t rank, cnt, base, counts, ret, tiles, tret, sched, order, seg, exp, iu, id, meta, flags, bands, trace,
        cslot, yrow, tcrow, bitem, tokof, xrows, xready, bytes;
};

StaticLayout static_layout(const Layout& lay) {
    const moe_layout& L = lay.L;
    const Shape& S = lay.S;
    StaticLayout o{};
    size_t cur = 0;
    auto put = [&](size_t bytes) {
        const size_t at = cur;
        cur = align_up(cur + bytes, 256);
        return at;
    };
    const size_t TK = (size_t)S.T * S.k, E = S.E, R = S.R, MT = L.MT_max;
    o.rank = put(TK * 4);
    o.cnt = put((size_t)L.n_chunks * E * 4);
    o.base = put((size_t)L.n_chunks * E * 4);
    o.counts = put(E * R * 4);
    o.ret = put(R * (E + 1) * 4);
    o.tiles = put(MT * 16);
    o.tret = put(MT * 4);
    o.sched = put(MT * 4);
    o.order = put(MT * 4);
    o.seg = put(MT * 8);
    o.exp = put(E * 32);
    o.iu = put((size_t)L.IU_max * 8);
    o.id = put(MT * 8);
    o.meta = put(META_COUNT * 4);
    o.flags = put(MT * (size_t)L.n_tiles_n2 * 4);
    o.bands = put(MT * 4);
    o.trace = put(TR_COUNT * 8);
    o.cslot = put(TK * 4);
    o.yrow = put((size_t)L.PC_max * 4);
    o.tcrow = put(MT * 4);
    o.bitem = put(MT * 4);
    o.tokof = put((size_t)L.PC_max * 4);
    o.xrows = put(E * 4);
    o.xready = put(E * 4);
    o.bytes = cur;
    return o;
}

// Device address of g_static_scratch in the current CUDA context. It is looked up once per context
// (a context made after cudaDeviceReset loads the module again, at another address) and cached by
// the context's process-unique id; without that id (an old driver) it is looked up on every call.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<Fn>(p);
    return nullptr;
}

constexpr int kStaticCache = 64;
std::mutex g_static_mu;
unsigned long long g_static_ctx[kStaticCache] = {};
void* g_static_addr[kStaticCache] = {};
int g_static_used = 0;

int static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);  // makes the device's primary context current
    if (e != cudaSuccess) return cuda_fail(e, "selecting the current device");
    static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 12000);
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    const bool keyed = get_ctx && get_id && get_ctx(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (keyed)
        for (int i = 0; i < g_static_used; ++i)
            if (g_static_ctx[i] == id) {
                *out = g_static_addr[i];
                return MOE_OK;
            }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
    if (keyed && g_static_used < kStaticCache) {
        g_static_ctx[g_static_used] = id;
        g_static_addr[g_static_used] = p;
        ++g_static_used;
    }
    *out = p;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

MOE_API int moe_workspace_size(const moe_config* cfg, size_t* bytes) {
    g_err.clear();
    if (!bytes) return fail(MOE_ERR_ARG, "bytes is NULL");
    Layout lay;
    const int rc = make_layout(cfg, &lay);
    if (rc) return rc;
    *bytes = lay.L.bytes;
    return MOE_OK;
}

MOE_API int moe_workspace_layout(const moe_config* cfg, moe_layout* out) {
    g_err.clear();
    if (!out) return fail(MOE_ERR_ARG, "out is NULL");
    Layout lay;
    const int rc = make_layout(cfg, &lay);
    if (rc) return rc;
    *out = lay.L;
    return MOE_OK;
}

MOE_API int moe_plan(const moe_config* cfg, const float* logits, const uint16_t* x, int32_t* topk_idx, float* topk_w,
                     void* ws, size_t ws_bytes, void* stream) {
    Call c;
    int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    const bool permute = !(cfg->flags & MOE_PLAN_SKIP_PERMUTE);
    if (!logits) return fail(MOE_ERR_ARG, "logits is NULL");
    if (permute && (!x || !aligned(x, 16))) return fail(MOE_ERR_ARG, "x must be non-NULL and 16-byte aligned");
    rc = run_plan(c, logits, x, permute);
    if (rc) return rc;
    const size_t tk = (size_t)cfg->T * cfg->topk;
    if (topk_idx) {
        cudaError_t e = cudaMemcpyAsync(topk_idx, c.p.idx, tk * 4, cudaMemcpyDeviceToDevice, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "copy of topk_idx");
    }
    if (topk_w) {
        cudaError_t e = cudaMemcpyAsync(topk_w, c.p.gate, tk * 4, cudaMemcpyDeviceToDevice, c.st);
        if (e != cudaSuccess) return cuda_fail(e, "copy of topk_w");
    }
    return MOE_OK;
}

MOE_API int moe_forward(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                        const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes, void* stream) {
    Call c;
    const int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    return run_forward(c, logits, x, W1, W3, W2, out, true);
}

MOE_API int moe_forward_sequential(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                                   const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes,
                                   void* stream) {
    Call c;
    const int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    return run_forward(c, logits, x, W1, W3, W2, out, false);
}

MOE_API int moe_copy_only(const moe_config* cfg, void* ws, size_t ws_bytes, int ctas, void* stream) {
    Call c;
    const int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    if (ctas < 1 || ctas > c.di.sms) return fail(MOE_ERR_ARG, "ctas=%d must be in [1, %d]", ctas, c.di.sms);
    cudaError_t e = cudaMemsetAsync(c.p.meta + META_QUEUE_SEQ, 0, sizeof(int32_t), c.st);
    if (e == cudaSuccess) e = launch_copy_seq(c.lay.S, c.p, ctas, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "copy-only launch");
    return MOE_OK;
}

MOE_API int moe_forward_ex(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                           const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes, int sequential,
                           void* const* stage_events, void* stream) {
    Call c;
    const int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    return run_forward(c, logits, x, W1, W3, W2, out, sequential == 0, stage_events);
}

MOE_API int moe_forward_host(const moe_config* cfg, const float* logits_h, const uint16_t* x_h, const uint16_t* W1,
                             const uint16_t* W3, const uint16_t* W2, float* out_h, void* ws, size_t ws_bytes,
                             int sequential, void* stream) {
    Call c;
    int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    if (!logits_h || !x_h || !out_h) return fail(MOE_ERR_ARG, "NULL host pointer");
    uint8_t* b = static_cast<uint8_t*>(ws);
    float* d_logits = reinterpret_cast<float*>(b + c.lay.L.in_logits);
    uint16_t* d_x = reinterpret_cast<uint16_t*>(b + c.lay.L.in_x);
    float* d_out = reinterpret_cast<float*>(b + c.lay.L.out);
    const size_t T = cfg->T;
    cudaError_t e = cudaMemcpyAsync(d_logits, logits_h, T * cfg->E * 4, cudaMemcpyHostToDevice, c.st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_x, x_h, T * cfg->d * 2, cudaMemcpyHostToDevice, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy of the inputs");
    rc = run_forward(c, d_logits, d_x, W1, W3, W2, d_out, sequential == 0);
    if (rc) return rc;
    e = cudaMemcpyAsync(out_h, d_out, T * cfg->d * 4, cudaMemcpyDeviceToHost, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy of the output");
    return MOE_OK;
}

// Internal copy streams and events of the pipelined host entry, created once per device.
// The layer's launches for one staging slot, captured once as a CUDA graph and replayed per batch
// (the tensor maps and pointers are fixed for a given config, workspace and weights).
struct LayerGraph {
    moe_config cfg;
    const void *ws, *W1, *W3, *W2;
    int sequential;
    cudaGraphExec_t exec[2];
    bool valid = false;
};
constexpr int LAYER_GRAPHS = 4;  // cached per device, oldest replaced first

struct HostPipe {
    cudaStream_t cin = nullptr, cout = nullptr, cap = nullptr;
    cudaEvent_t in_done[2], out_ready[2], out_free[2], slot_free[2];
    LayerGraph graphs[LAYER_GRAPHS];
    int next_graph = 0;
    bool ok = false;
};

static int host_pipe(HostPipe** out) {
    static HostPipe pipes[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_DEVICE, "device index %d out of range", dev);
    HostPipe& h = pipes[dev];
    if (!h.ok) {
        e = cudaStreamCreateWithFlags(&h.cin, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.cout, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.cap, cudaStreamNonBlocking);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&h.in_done[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.out_ready[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.out_free[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.slot_free[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return cuda_fail(e, "creating the copy streams and events");
        h.ok = true;
    }
    *out = &h;
    return MOE_OK;
}

// Graphs of the layer for the two staging slots of (cfg, ws, weights, sequential), captured on the
// pipe's capture stream at first use. Returns nullptr (and the caller launches eagerly) if the
// capture fails.
static const LayerGraph* layer_graphs(HostPipe* h, const Call& c, const moe_config* cfg, void* ws, const uint16_t* W1,
                                      const uint16_t* W3, const uint16_t* W2, int sequential) {
    for (const LayerGraph& g : h->graphs)
        if (g.valid && g.ws == ws && g.W1 == W1 && g.W3 == W3 && g.W2 == W2 && g.sequential == sequential &&
            memcmp(&g.cfg, cfg, sizeof(moe_config)) == 0)
            return &g;
    LayerGraph& g = h->graphs[h->next_graph];
    if (g.valid) {
        for (int sl = 0; sl < 2; ++sl) cudaGraphExecDestroy(g.exec[sl]);
        g.valid = false;
    }
    uint8_t* b = static_cast<uint8_t*>(ws);
    const size_t T = cfg->T, nl = T * cfg->E * 4, nx = T * cfg->d * 2, no = T * cfg->d * 4;
    Call cc = c;
    cc.st = h->cap;
    for (int sl = 0; sl < 2; ++sl) {
        cudaGraph_t graph = nullptr;
        if (cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return nullptr;
        const int rc = run_forward(cc, reinterpret_cast<const float*>(b + c.lay.L.in_logits + sl * nl),
                                   reinterpret_cast<const uint16_t*>(b + c.lay.L.in_x + sl * nx), W1, W3, W2,
                                   reinterpret_cast<float*>(b + c.lay.L.out + sl * no), sequential == 0);
        const cudaError_t e = cudaStreamEndCapture(h->cap, &graph);
        cudaGraphExec_t exec = nullptr;
        const bool ok = rc == MOE_OK && e == cudaSuccess && graph &&
                        cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
        if (graph) cudaGraphDestroy(graph);
        if (!ok) {
            if (sl == 1) cudaGraphExecDestroy(g.exec[0]);
            cudaGetLastError();  // the eager path reports its own errors
            g_err.clear();
            return nullptr;
        }
        g.exec[sl] = exec;
    }
    g.cfg = *cfg;
    g.ws = ws;
    g.W1 = W1;
    g.W3 = W3;
    g.W2 = W2;
    g.sequential = sequential;
    g.valid = true;
    h->next_graph = (h->next_graph + 1) % LAYER_GRAPHS;
    return &g;
}

MOE_API int moe_forward_host_pipelined(const moe_config* cfg, int steps, const float* const* logits_h,
                                       const uint16_t* const* x_h, const uint16_t* W1, const uint16_t* W3,
                                       const uint16_t* W2, float* const* out_h, void* ws, size_t ws_bytes,
                                       int sequential, void* stream) {
    Call c;
    int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    if (steps < 0) return fail(MOE_ERR_ARG, "steps=%d must be >= 0", steps);
    if (steps > 0 && (!logits_h || !x_h || !out_h)) return fail(MOE_ERR_ARG, "NULL host pointer array");
    for (int i = 0; i < steps; ++i)
        if (!logits_h[i] || !x_h[i] || !out_h[i]) return fail(MOE_ERR_ARG, "NULL host pointer (step %d)", i);
    HostPipe* h = nullptr;
    if ((rc = host_pipe(&h))) return rc;
    const LayerGraph* lg = steps > 1 ? layer_graphs(h, c, cfg, ws, W1, W3, W2, sequential) : nullptr;
    uint8_t* b = static_cast<uint8_t*>(ws);
    const size_t T = cfg->T, nl = T * cfg->E * 4, nx = T * cfg->d * 2, no = T * cfg->d * 4;
    cudaError_t e = cudaSuccess;
    // slot s of step i: its inputs go in after the layer of step i-2 (which read slot s) is done; its
    // layer waits for them and for the copy-out of step i-2 (which read slot s's output)
    for (int i = 0; i < steps && e == cudaSuccess; ++i) {
        const int sl = i & 1;
        float* d_logits = reinterpret_cast<float*>(b + c.lay.L.in_logits + sl * nl);
        uint16_t* d_x = reinterpret_cast<uint16_t*>(b + c.lay.L.in_x + sl * nx);
        float* d_out = reinterpret_cast<float*>(b + c.lay.L.out + sl * no);
        if (i == 0) e = cudaEventRecord(h->slot_free[0], c.st);  // the caller's earlier work on the workspace
        if (i == 0 && e == cudaSuccess) e = cudaEventRecord(h->slot_free[1], c.st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->cin, h->slot_free[sl], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(d_logits, logits_h[i], nl, cudaMemcpyHostToDevice, h->cin);
        if (e == cudaSuccess) e = cudaMemcpyAsync(d_x, x_h[i], nx, cudaMemcpyHostToDevice, h->cin);
        if (e == cudaSuccess) e = cudaEventRecord(h->in_done[sl], h->cin);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c.st, h->in_done[sl], 0);
        if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(c.st, h->out_free[sl], 0);
        if (e != cudaSuccess) break;
        if (lg) {
            e = cudaGraphLaunch(lg->exec[sl], c.st);
            if (e != cudaSuccess) break;
        } else {
            rc = run_forward(c, d_logits, reinterpret_cast<const uint16_t*>(d_x), W1, W3, W2, d_out,
                             sequential == 0);
            if (rc) return rc;
        }
        e = cudaEventRecord(h->out_ready[sl], c.st);
        if (e == cudaSuccess) e = cudaEventRecord(h->slot_free[sl], c.st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->cout, h->out_ready[sl], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(out_h[i], d_out, no, cudaMemcpyDeviceToHost, h->cout);
        if (e == cudaSuccess) e = cudaEventRecord(h->out_free[sl], h->cout);
    }
    // the caller's stream reaches the end of this call only after every copy-out
    for (int sl = 0; sl < 2 && e == cudaSuccess && steps > sl; ++sl) e = cudaStreamWaitEvent(c.st, h->out_free[sl], 0);
    if (e != cudaSuccess) return cuda_fail(e, "pipelined host copies");
    return MOE_OK;
}

// ---- copy-engine return copy (moe_forward_dma) ------------------------------------------------
// The return copy on the GPU's copy engines: the down-projection runs on every SM without consumers,
// and the epilogue warp that completes a band writes a record into pinned host memory (Yp row, Ret
// row, valid rows, then the call's tag, released at system scope). The calling thread polls the
// records and issues one cudaMemcpyAsync per run of ready bands that are adjacent in both Yp and Ret
// (else per band) on a copy stream of its own; the combine
// waits for that stream. Records: 4 words of header (tag, band count, padded rows, 0), then 4 words
// per band (tag, Ret row, valid rows, Yp row).
struct DmaPipe {
    cudaStream_t cs = nullptr;
    cudaEvent_t start = nullptr, copied = nullptr;
    bool ok = false;
};

static int dma_pipe(DmaPipe** out) {
    static DmaPipe pipes[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    DmaPipe& d = pipes[dev];
    if (!d.ok) {
        e = cudaStreamCreateWithFlags(&d.cs, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.copied, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "creating the copy-engine stream and events");
        d.ok = true;
    }
    *out = &d;
    return MOE_OK;
}

static size_t dma_host_bytes(const Layout& lay) { return (size_t)(lay.L.MT_max + 1) * 16; }

static int run_forward_dma(Call& c, const float* logits, const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                           const uint16_t* W2, float* out, void* host_rec, size_t host_bytes, void* const* ev) {
    if (!logits || !x || !W1 || !W3 || !W2 || !out) return fail(MOE_ERR_ARG, "NULL input or output pointer");
    if (!aligned(x, 16) || !aligned(W1, 16) || !aligned(W3, 16) || !aligned(W2, 16) || !aligned(out, 16) ||
        !aligned(logits, 4))
        return fail(MOE_ERR_ARG, "x, W1, W3, W2, out must be 16-byte aligned, logits 4-byte aligned");
    if (!host_rec || !aligned(host_rec, 16)) return fail(MOE_ERR_ARG, "host_rec must be non-NULL and 16-byte aligned");
    if (host_bytes < dma_host_bytes(c.lay))
        return fail(MOE_ERR_ARG, "host_rec has %zu bytes, needs %zu", host_bytes, dma_host_bytes(c.lay));
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(c.st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(MOE_ERR_ARG, "moe_forward_dma waits on the host for the GPU: it cannot be captured in a graph");
    void* dev_rec = nullptr;
    e = cudaHostGetDevicePointer(&dev_rec, host_rec, 0);
    if (e != cudaSuccess) return cuda_fail(e, "host_rec is not pinned memory mapped into the device");
    DmaPipe* dp = nullptr;
    int rc = dma_pipe(&dp);
    if (rc) return rc;

    // no consumer SMs: the down-projection on every SM, flags published, nothing copied by SMs
    static std::atomic<uint32_t> g_epoch{0};
    uint32_t epoch = ++g_epoch;
    if (epoch == 0) epoch = ++g_epoch;
    Shape& S = c.lay.S;
    S.flags &= ~(uint32_t)(MOE_TAIL_ASSIST | MOE_COPY_WARPS | MOE_ADAPTIVE_CONSUMERS | MOE_TEST_STALL_CONSUMER);
    S.host_epoch = epoch;
    c.p.host_rec = static_cast<uint32_t*>(dev_rec);
    const bool pair_down = (S.flags & MOE_PAIR_UMMA) && S.bn2 == 2 * BN1;
    CUtensorMap tXc, tHc, tW1, tW3, tW2, tW2h, tHcOut, tYpOut;
    rc = make_map(&tXc, c.p.Xc, 2, S.d, S.PC_max, 1, BM, "Xc");
    if (!rc) rc = make_map(&tHc, c.p.Hc, 2, S.ffn, S.PC_max, 1, BM, "Hc");
    if (!rc) rc = make_map(&tHcOut, c.p.Hc, 2, S.ffn, S.PC_max, 1, 32, "Hc (store)", EPI_CHUNK, false);
    if (!rc) rc = make_map(&tYpOut, c.p.Yp, 2, S.d, S.P_max, 1, 32, "Yp (store)", EPI_CHUNK, false);
    if (!rc) rc = make_map(&tW1, W1, 3, S.d, S.ffn, S.E, BN1, "W1");
    if (!rc) rc = make_map(&tW3, W3, 3, S.d, S.ffn, S.E, BN1, "W3");
    if (!rc) rc = make_map(&tW2, W2, 3, S.ffn, S.d, S.E, S.bn2, "W2");
    if (!rc && pair_down) rc = make_map(&tW2h, W2, 3, S.ffn, S.d, S.E, BN1, "W2 (half)");
    if (rc) return rc;

    // the copy stream starts after everything the caller enqueued before (the last combine read Ret)
    e = cudaEventRecord(dp->start, c.st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(dp->cs, dp->start, 0);
    if (e != cudaSuccess) return cuda_fail(e, "ordering the copy stream");
    if ((rc = record(ev, MOE_EV_BEGIN, c.st))) return rc;
    c.p.x = reinterpret_cast<const __nv_bfloat16*>(x);
    if ((rc = run_plan(c, logits, x, !(S.flags & MOE_FUSED_DISPATCH)))) return rc;
    if ((rc = record(ev, MOE_EV_PLANNED, c.st))) return rc;
    e = (S.flags & MOE_PAIR_UMMA) ? launch_gemm_swiglu_pair(S, c.p, tXc, tW1, tW3, tHcOut, c.st)
                                  : launch_gemm_swiglu(S, c.p, tXc, tW1, tW3, tHcOut, c.di.sms, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "SwiGLU GEMM launch");
    if ((rc = record(ev, MOE_EV_UP, c.st))) return rc;
    e = pair_down ? launch_gemm_down_pair(S, c.p, tHc, tW2h, tYpOut, 0, true, c.st)
                  : launch_gemm_down(S, c.p, tHc, tW2, tYpOut, c.di.sms, 0, true, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "down-projection launch");
    if ((rc = record(ev, MOE_EV_DOWN, c.st))) return rc;

    // Poll the records; a band's copy is issued as soon as its record carries this call's tag. The
    // wait needs no time limit: once the main stream has run everything enqueued (its last kernel is
    // the down-projection), every record of the call has been written, so a scan after that which
    // still misses one is an error (a kernel stopped early), not a reason to wait longer.
    volatile uint32_t* h = static_cast<volatile uint32_t*>(host_rec);
    const size_t rowb = (size_t)S.d * 2;
    uint8_t* Yp = reinterpret_cast<uint8_t*>(c.p.Yp);
    uint8_t* Ret = reinterpret_cast<uint8_t*>(c.p.Ret);
    int MT = -1, issued = 0;
    std::vector<char> done;
    bool drained = false;  // the main stream had finished before the current scan began
    for (uint64_t it = 0;; ++it) {
        const bool last_scan = drained;
        if (MT < 0 && h[0] == epoch) {
            std::atomic_thread_fence(std::memory_order_acquire);
            MT = (int)h[1];
            if (MT < 0 || MT > S.MT_max) return fail(MOE_ERR_PLAN, "band count %d out of range", MT);
            done.assign((size_t)MT, 0);
        }
        // Ready bands that are adjacent in both Yp and Ret (a group's bands in layout order) go out as
        // one copy: one host call per run instead of per band.
        uint32_t run_ret = 0, run_row = 0, run_rows = 0;
        auto flush = [&]() -> int {
            if (run_rows == 0) return MOE_OK;
            const cudaError_t ce = cudaMemcpyAsync(Ret + (size_t)run_ret * rowb, Yp + (size_t)run_row * rowb,
                                                   run_rows * rowb, cudaMemcpyDeviceToDevice, dp->cs);
            run_rows = 0;
            return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "copy-engine band copy");
        };
        for (int m = 0; MT > 0 && m < MT; ++m) {
            if (done[m] || h[4 + 4 * (size_t)m] != epoch) {
                if ((rc = flush())) return rc;
                continue;
            }
            std::atomic_thread_fence(std::memory_order_acquire);
            const uint32_t ret0 = h[4 + 4 * (size_t)m + 1], valid = h[4 + 4 * (size_t)m + 2],
                           row0 = h[4 + 4 * (size_t)m + 3];
            if (valid > (uint32_t)S.tbM || (size_t)ret0 + valid > (size_t)S.T * S.k ||
                (size_t)row0 + valid > (size_t)S.P_max)
                return fail(MOE_ERR_PLAN, "band %d record out of range", m);
            if (valid == 0) {  // returned by the down-projection's epilogue (MOE_DIRECT_TAIL)
                if ((rc = flush())) return rc;
                done[m] = 1;
                ++issued;
                continue;
            }
            if (run_rows && (ret0 != run_ret + run_rows || row0 != run_row + run_rows) && (rc = flush())) return rc;
            if (run_rows == 0) {
                run_ret = ret0;
                run_row = row0;
            }
            run_rows += valid;
            done[m] = 1;
            ++issued;
        }
        if ((rc = flush())) return rc;
        if (MT >= 0 && issued == MT) break;
        if (last_scan) {
            if (MT < 0) return fail(MOE_ERR_PLAN, "the plan kernel finished without its host record");
            return fail(MOE_ERR_TIMEOUT, "the down-projection finished with %d of %d band records (see moe_status)",
                        issued, MT);
        }
        if ((it & 15) == 15) {
            e = cudaStreamQuery(c.st);
            if (e == cudaSuccess) drained = true;  // one more scan, then every record must be there
            else if (e != cudaErrorNotReady) return cuda_fail(e, "main stream");
        }
    }
    if ((rc = record(ev, MOE_EV_COPIED, dp->cs))) return rc;
    e = cudaEventRecord(dp->copied, dp->cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c.st, dp->copied, 0);
    if (e != cudaSuccess) return cuda_fail(e, "joining the copy stream");
    e = launch_combine(S, c.p, out, c.di.sms, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return record(ev, MOE_EV_END, c.st);
}

MOE_API int moe_dma_host_bytes(const moe_config* cfg, size_t* bytes) {
    g_err.clear();
    if (!bytes) return fail(MOE_ERR_ARG, "bytes is NULL");
    Layout lay;
    const int rc = make_layout(cfg, &lay);
    if (rc) return rc;
    *bytes = dma_host_bytes(lay);
    return MOE_OK;
}

MOE_API int moe_forward_dma(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes,
                            void* host_rec, size_t host_bytes, void* const* stage_events, void* stream) {
    Call c;
    const int rc = begin_call(cfg, ws, ws_bytes, stream, &c);
    if (rc) return rc;
    return run_forward_dma(c, logits, x, W1, W3, W2, out, host_rec, host_bytes, stage_events);
}

MOE_API int moe_status(const moe_config* cfg, const void* ws, void* stream, int32_t* detail) {
    g_err.clear();
    Layout lay;
    int rc = make_layout(cfg, &lay);
    if (rc) return rc;
    // ws == NULL: the status words of the last moe_route_static call, in the static scratch
    const uint8_t* meta = nullptr;
    if (ws) {
        meta = static_cast<const uint8_t*>(ws) + lay.L.meta;
    } else {
        const StaticLayout o = static_layout(lay);
        if (o.bytes > (size_t)MOE_STATIC_SCRATCH_BYTES)
            return fail(MOE_ERR_ARG, "this config does not fit the static scratch (%zu bytes)", o.bytes);
        void* base = nullptr;
        if ((rc = static_scratch(&base))) return rc;
        meta = static_cast<const uint8_t*>(base) + o.meta;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int32_t w[2] = {0, 0};
    e = cudaMemcpy(w, meta + META_STATUS * 4, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (detail) *detail = w[1];
    switch (w[0]) {
        case ST_OK: return MOE_OK;
        case ST_FLAG_TIMEOUT: return fail(MOE_ERR_TIMEOUT, "consumer flag wait timed out (M-tile %d)", w[1]);
        case ST_PIPE_TIMEOUT: return fail(MOE_ERR_TIMEOUT, "GEMM pipeline wait timed out (role %d)", w[1]);
        case ST_COPY_TIMEOUT: return fail(MOE_ERR_TIMEOUT, "row-band copy timed out (M-tile %d)", w[1]);
        case ST_BAD_PLAN: return fail(MOE_ERR_PLAN, "plan index out of bounds (%d)", w[1]);
        case ST_PAIR_TMEM: return fail(MOE_ERR_DEVICE, "CTA pair got different TMEM bases (peer %d)", w[1]);
        case ST_LAYOUT_TIMEOUT: return fail(MOE_ERR_TIMEOUT, "permute's wait for the row layout timed out");
        default: return fail(MOE_ERR_PLAN, "unknown device status %d", w[0]);
    }
}

MOE_API int moe_device_info(int32_t* sm_count, int32_t* supported) {
    g_err.clear();
    DeviceInfo di;
    const int rc = device_info(&di);
    if (rc) return rc;
    if (sm_count) *sm_count = di.sms;
    if (supported) *supported = di.supported ? 1 : 0;
    return MOE_OK;
}

MOE_API int moe_route_static(const moe_config* cfg, const float* logits, int32_t* topk_idx, float* topk_w,
                             int32_t* slot, int32_t* ret_slot, int32_t* offsets, void* stream) {
    g_err.clear();
    Layout lay;
    int rc = make_layout(cfg, &lay);
    if (rc) return rc;
    if (!logits || !topk_idx || !topk_w || !slot || !ret_slot || !offsets)
        return fail(MOE_ERR_ARG, "NULL input or output pointer");
    const StaticLayout o = static_layout(lay);
    if (o.bytes > (size_t)MOE_STATIC_SCRATCH_BYTES)
        return fail(MOE_ERR_ARG, "this config needs %zu bytes of static scratch; the limit is %d", o.bytes,
                    MOE_STATIC_SCRATCH_BYTES);
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    if (!di.supported) return fail(MOE_ERR_DEVICE, "current device is not sm_103 (GB300)");
    void* base = nullptr;
    if ((rc = static_scratch(&base))) return rc;
    uint8_t* b = static_cast<uint8_t*>(base);
    PlanPtrs p{};
    p.idx = topk_idx;
    p.gate = topk_w;
    p.rank = reinterpret_cast<int32_t*>(b + o.rank);
    p.chunk_cnt = reinterpret_cast<int32_t*>(b + o.cnt);
    p.chunk_base = reinterpret_cast<int32_t*>(b + o.base);
    p.counts = reinterpret_cast<int32_t*>(b + o.counts);
    p.offsets = offsets;
    p.ret_off = reinterpret_cast<int32_t*>(b + o.ret);
    p.tiles = reinterpret_cast<int32_t*>(b + o.tiles);
    p.tile_ret = reinterpret_cast<int32_t*>(b + o.tret);
    p.sched = reinterpret_cast<int32_t*>(b + o.sched);
    p.order = reinterpret_cast<int32_t*>(b + o.order);
    p.seg = reinterpret_cast<int32_t*>(b + o.seg);
    p.experts = reinterpret_cast<int32_t*>(b + o.exp);
    p.items_up = reinterpret_cast<int32_t*>(b + o.iu);
    p.items_down = reinterpret_cast<int32_t*>(b + o.id);
    p.slot = slot;
    p.cslot = reinterpret_cast<int32_t*>(b + o.cslot);
    p.ret_slot = ret_slot;
    p.yrow = reinterpret_cast<int32_t*>(b + o.yrow);
    p.tile_crow = reinterpret_cast<int32_t*>(b + o.tcrow);
    p.band_item = reinterpret_cast<int32_t*>(b + o.bitem);
    p.tok_of = reinterpret_cast<int32_t*>(b + o.tokof);
    p.xrows = reinterpret_cast<uint32_t*>(b + o.xrows);
    p.xready = reinterpret_cast<uint32_t*>(b + o.xready);
    p.meta = reinterpret_cast<int32_t*>(b + o.meta);
    p.flags = reinterpret_cast<uint32_t*>(b + o.flags);
    p.bands = reinterpret_cast<uint32_t*>(b + o.bands);
    p.trace = reinterpret_cast<unsigned long long*>(b + o.trace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the plan-only kernels: no token rows are moved (x = NULL), whatever cfg->flags says
    lay.S.flags &= MOE_TEST_PLAN_FAIL;
    cudaError_t e = launch_route(lay.S, logits, p, st);
    if (e == cudaSuccess) e = launch_plan(lay.S, p, st);
    if (e == cudaSuccess) e = launch_permute(lay.S, nullptr, p, di.sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "static-scratch plan launch");
    return MOE_OK;
}

MOE_API const char* moe_last_error(void) { return g_err.c_str(); }

}  // extern "C"
