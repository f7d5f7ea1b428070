// hq_api.cu -- the C ABI declared in include/hq.h: argument validation, error
// reporting, per-device set-up, and dispatch to the kernels.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <cmath>

#include "hq_internal.h"

namespace hq {

// The fault word that kernels set instead of trapping (see hq.h).
__device__ uint32_t g_fault_word;

// Scratch of hq_matvec_q8_0_lora_noalloc, the QLoRA call for callers that
// cannot allocate device memory: u = A x for the largest adapter (rank 64) at
// the widest call (8 vectors), 2 KB.  One per device, in the module's static
// device memory, held until the process exits.  In host code the symbol is a
// host-side stand-in, so device_info() looks up its device address once per
// device (with that device current) and launches use that address.
constexpr int kNoAllocScratchFloats = 64 * 8;
static __device__ __align__(256) float g_lora_scratch[kNoAllocScratchFloats];

namespace {

thread_local char t_error[512] = "";
std::mutex g_mutex;
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
// g_ready[d] == d + 1 once g_devices[d] is complete: written (release) after
// the record under g_mutex, read (acquire) before the record without it.
std::atomic<int> g_ready[kMaxDevices];
void *g_encoder = nullptr;
bool g_encoder_tried = false;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

hq_status set_error(hq_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_error, sizeof(t_error), fmt, ap);
    va_end(ap);
    return st;
}

hq_status device_info(DeviceInfo **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(HQ_ERR_UNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_error(HQ_ERR_UNSUPPORTED, "device index %d too large", dev);
    DeviceInfo &d = g_devices[dev];
    if (g_ready[dev].load(std::memory_order_acquire) == dev + 1) { *out = &d; return HQ_OK; }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_ready[dev].load(std::memory_order_relaxed) != dev + 1) {
        DeviceInfo n;
        n.device = dev;
        if (cudaDeviceGetAttribute(&n.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return set_error(HQ_ERR_UNSUPPORTED, "cudaDeviceGetAttribute failed");
        if (n.cc_major != 10 || n.cc_minor != 3)
            return set_error(HQ_ERR_UNSUPPORTED, "built for sm_103a; device %d is sm_%d%d", dev, n.cc_major, n.cc_minor);
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fault_word);
        if (e != cudaSuccess) return set_error(HQ_ERR_UNSUPPORTED, "fault word: %s", cudaGetErrorString(e));
        n.fault = static_cast<uint32_t *>(p);
        e = cudaGetSymbolAddress(&p, g_lora_scratch);
        if (e != cudaSuccess) return set_error(HQ_ERR_UNSUPPORTED, "adapter scratch: %s", cudaGetErrorString(e));
        n.lora_scratch = static_cast<float *>(p);
        d = n;
        g_ready[dev].store(dev + 1, std::memory_order_release);
    }
    *out = &d;
    return HQ_OK;
}

void *tensor_map_encoder() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encoder_tried) {
        g_encoder_tried = true;
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encoder = fn;
    }
    return g_encoder;
}


std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace hq

using namespace hq;

namespace {

hq_status check_float_matvec(const void *W, const float *x, float *y, int64_t rows, int64_t cols, int n_vec) {
    if (!W || !x || !y) return set_error(HQ_ERR_NULL, "W, x and y must be non-null");
    if (n_vec < 1 || n_vec > 8) return set_error(HQ_ERR_NVEC, "n_vec %d not in [1,8]", n_vec);
    if (rows < 1 || rows > 0x7fffffffLL || cols < 32 || cols % 32 != 0 || cols > (1LL << 31))
        return set_error(HQ_ERR_SHAPE, "bad shape rows=%lld cols=%lld (need rows>=1, cols>=32, cols%%32==0)",
                         (long long)rows, (long long)cols);
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4))
        return set_error(HQ_ERR_ALIGN, "W and x must be 16-byte aligned, y 4-byte aligned");
    return HQ_OK;
}

hq_status finish(hq_status st) {
    if (st == HQ_OK) t_error[0] = '\0';
    return st;
}

}  // namespace

extern "C" {

int hq_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char *hq_last_error(void) { return t_error; }

hq_status hq_matvec_q8_0(const void *W, const float *x, float *y, int64_t rows, int64_t cols,
                         int n_vec, hq_stream_t stream) {
    hq_status st = check_float_matvec(W, x, y, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    return finish(launch_matvec_float_q8_0(W, x, y, rows, cols, n_vec, nullptr, (cudaStream_t)stream));
}

hq_status hq_matvec_q4_0(const void *W, const float *x, float *y, int64_t rows, int64_t cols,
                         int n_vec, hq_stream_t stream) {
    hq_status st = check_float_matvec(W, x, y, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    return finish(launch_matvec_float_q4_0(W, x, y, rows, cols, n_vec, nullptr, (cudaStream_t)stream));
}

hq_status hq_matvec_q4_k(const void *W, const float *x, float *y, int64_t rows, int64_t cols,
                         int n_vec, hq_stream_t stream) {
    hq_status st = check_float_matvec(W, x, y, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    if (cols % 256 != 0) return set_error(HQ_ERR_SHAPE, "Q4_K needs cols %% 256 == 0 (cols = %lld)", (long long)cols);
    return finish(launch_matvec_float_q4_k(W, x, y, rows, cols, n_vec, nullptr, (cudaStream_t)stream));
}

// The float matvec plus the QLoRA adapter term: u = A x into the caller's
// workspace, then the matvec adds scale * B u as it stores each output.
static hq_status matvec_lora(int fmt, const void *W, const float *x, const uint16_t *A, const uint16_t *B,
                             float scale, int rank, float *workspace, float *y, int64_t rows, int64_t cols,
                             int n_vec, hq_stream_t stream) {
    hq_status st = check_float_matvec(W, x, y, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    if (!A || !B || !workspace) return set_error(HQ_ERR_NULL, "lora_A, lora_B and workspace must be non-null");
    if (rank < 1 || rank > 64) return set_error(HQ_ERR_SHAPE, "rank %d not in [1,64]", rank);
    if (!std::isfinite(scale)) return set_error(HQ_ERR_SHAPE, "scale must be finite");
    if (!aligned(A, 16) || !aligned(B, 2) || !aligned(workspace, 4))
        return set_error(HQ_ERR_ALIGN, "lora_A must be 16-byte aligned, lora_B 2-byte, workspace 4-byte");
    cudaStream_t s = (cudaStream_t)stream;
    st = launch_lora_down(A, x, workspace, rank, cols, n_vec, s);
    if (st != HQ_OK) return st;
    MatvecExtras l;
    l.B = B;
    l.u = workspace;
    l.scale = scale;
    l.rank = rank;
    return finish(fmt == 8 ? launch_matvec_float_q8_0(W, x, y, rows, cols, n_vec, &l, s)
                           : launch_matvec_float_q4_0(W, x, y, rows, cols, n_vec, &l, s));
}

// hq_matvec_q8_0_lora with u = A x kept in the per-device static scratch
// instead of a caller's workspace: the call allocates and takes no memory.
// Calls that overlap on one device race on the scratch (see hq.h).
hq_status hq_matvec_q8_0_lora_noalloc(const void *W, const float *x, const uint16_t *lora_A,
                                      const uint16_t *lora_B, float scale, int rank, float *y, int64_t rows,
                                      int64_t cols, int n_vec, hq_stream_t stream) {
    // argument checks first, without touching a device
    hq_status st = check_float_matvec(W, x, y, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    if (!lora_A || !lora_B) return set_error(HQ_ERR_NULL, "lora_A and lora_B must be non-null");
    if (rank < 1 || rank > 64) return set_error(HQ_ERR_SHAPE, "rank %d not in [1,64]", rank);
    static_assert(kNoAllocScratchFloats >= 64 * 8, "scratch holds rank 64 x 8 vectors");
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != HQ_OK) return st;
    return matvec_lora(8, W, x, lora_A, lora_B, scale, rank, dev->lora_scratch, y, rows, cols, n_vec, stream);
}

uint64_t hq_launch_count(void) { return hq::g_launches.load(std::memory_order_relaxed); }

hq_status hq_debug_plan(int fmt, int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs,
                        int64_t *out, int out_len) {
    if (!out) return set_error(HQ_ERR_NULL, "out must be non-null");
    if (out_len < HQ_PLAN_FIELDS) return set_error(HQ_ERR_SHAPE, "out needs %d entries", HQ_PLAN_FIELDS);
    if (n_vec < 1 || n_vec > 8) return set_error(HQ_ERR_NVEC, "n_vec %d not in [1,8]", n_vec);
    if (rows < 1 || rows > 0x7fffffffLL) return set_error(HQ_ERR_SHAPE, "rows %lld out of range", (long long)rows);
    if (num_sms < 1 || smem_optin < 1024 || regs < 1 || regs > 255)
        return set_error(HQ_ERR_SHAPE, "device description out of range (num_sms %d, smem %d, regs %d)", num_sms,
                         smem_optin, regs);
    const int64_t chunk = fmt == 1 ? 128 : 256;
    if (cols < chunk || cols % chunk != 0 || cols > (1LL << 31))
        return set_error(HQ_ERR_SHAPE, "cols %lld: the staged kernel needs a multiple of %lld", (long long)cols,
                         (long long)chunk);
    switch (fmt) {
        case 8: return debug_plan_float_q8_0(n_vec, rows, cols, num_sms, smem_optin, regs, out);
        case 4: return debug_plan_float_q4_0(n_vec, rows, cols, num_sms, smem_optin, regs, out);
        case HQ_FMT_Q4_K: return debug_plan_float_q4_k(n_vec, rows, cols, num_sms, smem_optin, regs, out);
        case 1: return debug_plan_i8(n_vec, rows, cols, num_sms, smem_optin, regs, out);
        default: return set_error(HQ_ERR_UNSUPPORTED, "fmt %d: 8 (Q8_0), 4 (Q4_0), 75 (Q4_K) or 1 (int8)", fmt);
    }
}

hq_status hq_matvec_q8_0_lora(const void *W, const float *x, const uint16_t *lora_A, const uint16_t *lora_B,
                              float scale, int rank, float *workspace, float *y, int64_t rows, int64_t cols,
                              int n_vec, hq_stream_t stream) {
    return matvec_lora(8, W, x, lora_A, lora_B, scale, rank, workspace, y, rows, cols, n_vec, stream);
}

hq_status hq_matvec_q4_0_lora(const void *W, const float *x, const uint16_t *lora_A, const uint16_t *lora_B,
                              float scale, int rank, float *workspace, float *y, int64_t rows, int64_t cols,
                              int n_vec, hq_stream_t stream) {
    return matvec_lora(4, W, x, lora_A, lora_B, scale, rank, workspace, y, rows, cols, n_vec, stream);
}

hq_status hq_matvec_i8_requant(const int8_t *W, const int8_t *x, const int32_t *mult,
                               const int32_t *shift, int8_t *y, int64_t rows, int64_t cols, int n_vec,
                               hq_stream_t stream) {
    if (!W || !x || !mult || !shift || !y) return set_error(HQ_ERR_NULL, "W, x, mult, shift and y must be non-null");
    if (n_vec < 1 || n_vec > 8) return set_error(HQ_ERR_NVEC, "n_vec %d not in [1,8]", n_vec);
    if (rows < 1 || rows > 0x7fffffffLL || cols < 4 || cols % 4 != 0 || cols > (1LL << 31))
        return set_error(HQ_ERR_SHAPE, "bad shape rows=%lld cols=%lld (need rows>=1, cols>=4, cols%%4==0)",
                         (long long)rows, (long long)cols);
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(mult, 4) || !aligned(shift, 4))
        return set_error(HQ_ERR_ALIGN, "W and x must be 16-byte aligned, mult and shift 4-byte aligned");
    return finish(launch_matvec_i8(W, x, mult, shift, y, rows, cols, n_vec, (cudaStream_t)stream));
}

static hq_status check_moe(const void *W_bank, const int32_t *expert_ids, const float *x, int x_per_slot,
                           const float *y, int64_t n_experts, int n_active, int64_t rows, int64_t cols, int n_vec) {
    if (!W_bank || !expert_ids || !x || !y) return set_error(HQ_ERR_NULL, "W_bank, expert_ids, x and y must be non-null");
    if (n_vec < 1 || n_vec > 8) return set_error(HQ_ERR_NVEC, "n_vec %d not in [1,8]", n_vec);
    if (n_experts < 1 || n_active < 1 || n_active > n_experts || (long long)n_vec * n_active > 256 ||
        rows < 1 || cols < 256 || cols % 256 != 0 || rows * n_experts > 0x7fffffffLL || cols > (1LL << 31) ||
        (x_per_slot != 0 && x_per_slot != 1))
        return set_error(HQ_ERR_SHAPE,
                         "bad MoE shape n_experts=%lld n_active=%d rows=%lld cols=%lld x_per_slot=%d "
                         "(need 1<=n_active<=n_experts, n_vec*n_active<=256, cols%%256==0)",
                         (long long)n_experts, n_active, (long long)rows, (long long)cols, x_per_slot);
    if (!aligned(W_bank, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(expert_ids, 4))
        return set_error(HQ_ERR_ALIGN, "W_bank and x must be 16-byte aligned");
    return HQ_OK;
}

hq_status hq_moe_matvec_q8_0(const void *W_bank, const int32_t *expert_ids, const float *x,
                             int x_per_slot, float *y, int64_t n_experts, int n_active, int64_t rows,
                             int64_t cols, int n_vec, hq_stream_t stream) {
    hq_status st = check_moe(W_bank, expert_ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    return finish(launch_moe_q8_0(W_bank, expert_ids, x, x_per_slot, y, n_experts, n_active, rows, cols,
                                  n_vec, nullptr, (cudaStream_t)stream));
}

hq_status hq_moe_matvec_q8_0_swiglu(const void *W_bank, const int32_t *expert_ids, const float *x,
                                    int x_per_slot, float *h, int64_t n_experts, int n_active, int64_t rows,
                                    int64_t cols, int n_vec, hq_stream_t stream) {
    hq_status st = check_moe(W_bank, expert_ids, x, x_per_slot, h, n_experts, n_active, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    if (rows % 2 != 0)
        return set_error(HQ_ERR_SHAPE, "SwiGLU needs interleaved gate/up rows: rows = %lld is odd", (long long)rows);
    MoeEpi e;
    e.kind = 1;
    return finish(launch_moe_q8_0(W_bank, expert_ids, x, x_per_slot, h, n_experts, n_active, rows, cols,
                                  n_vec, &e, (cudaStream_t)stream));
}

hq_status hq_moe_matvec_q8_0_combine(const void *W_bank, const int32_t *expert_ids, const float *x,
                                     int x_per_slot, const float *router_w, float *y, int64_t n_experts,
                                     int n_active, int64_t rows, int64_t cols, int n_vec, hq_stream_t stream) {
    hq_status st = check_moe(W_bank, expert_ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    if (!router_w) return set_error(HQ_ERR_NULL, "router_w must be non-null");
    if (!aligned(router_w, 4)) return set_error(HQ_ERR_ALIGN, "router_w must be 4-byte aligned");
    MoeEpi e;
    e.kind = 2;
    e.router_w = router_w;
    return finish(launch_moe_q8_0(W_bank, expert_ids, x, x_per_slot, y, n_experts, n_active, rows, cols,
                                  n_vec, &e, (cudaStream_t)stream));
}

hq_status hq_moe_matvec_q8_0_ex(const void *W_bank, const int32_t *expert_ids, const float *x, int x_per_slot,
                                const float *router_w, float *y, int64_t n_experts, int n_active, int64_t rows,
                                int64_t cols, int n_vec, int epilogue, int flags, hq_stream_t stream) {
    hq_status st = check_moe(W_bank, expert_ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec);
    if (st != HQ_OK) return st;
    if (epilogue < HQ_MOE_EPI_NONE || epilogue > HQ_MOE_EPI_COMBINE)
        return set_error(HQ_ERR_UNSUPPORTED, "epilogue %d is not HQ_MOE_EPI_NONE, _SWIGLU or _COMBINE", epilogue);
    if (flags & ~HQ_MOE_IDS_READY) return set_error(HQ_ERR_UNSUPPORTED, "unknown flags %#x", flags);
    if (epilogue == HQ_MOE_EPI_SWIGLU && rows % 2 != 0)
        return set_error(HQ_ERR_SHAPE, "SwiGLU needs interleaved gate/up rows: rows = %lld is odd", (long long)rows);
    if (epilogue == HQ_MOE_EPI_COMBINE) {
        if (!router_w) return set_error(HQ_ERR_NULL, "router_w must be non-null");
        if (!aligned(router_w, 4)) return set_error(HQ_ERR_ALIGN, "router_w must be 4-byte aligned");
    }
    MoeEpi e;
    e.kind = epilogue;
    e.router_w = epilogue == HQ_MOE_EPI_COMBINE ? router_w : nullptr;
    e.ids_ready = (flags & HQ_MOE_IDS_READY) ? 1 : 0;
    return finish(launch_moe_q8_0(W_bank, expert_ids, x, x_per_slot, y, n_experts, n_active, rows, cols,
                                  n_vec, &e, (cudaStream_t)stream));
}

hq_status hq_quantize_q8_0(const float *W, void *out, int64_t rows, int64_t cols, hq_stream_t stream) {
    if (!W || !out) return set_error(HQ_ERR_NULL, "W and out must be non-null");
    if (rows < 1 || cols < 32 || cols % 32 != 0) return set_error(HQ_ERR_SHAPE, "need rows>=1, cols%%32==0");
    if (!aligned(W, 16) || !aligned(out, 2)) return set_error(HQ_ERR_ALIGN, "W must be 16-byte aligned");
    return finish(launch_quantize(0, W, out, nullptr, rows, cols, (cudaStream_t)stream));
}

hq_status hq_quantize_q4_0(const float *W, void *out, int64_t rows, int64_t cols, hq_stream_t stream) {
    if (!W || !out) return set_error(HQ_ERR_NULL, "W and out must be non-null");
    if (rows < 1 || cols < 32 || cols % 32 != 0) return set_error(HQ_ERR_SHAPE, "need rows>=1, cols%%32==0");
    if (!aligned(W, 16) || !aligned(out, 2)) return set_error(HQ_ERR_ALIGN, "W must be 16-byte aligned");
    return finish(launch_quantize(1, W, out, nullptr, rows, cols, (cudaStream_t)stream));
}

hq_status hq_quantize_q4_k(const float *W, void *out, int64_t rows, int64_t cols, hq_stream_t stream) {
    if (!W || !out) return set_error(HQ_ERR_NULL, "W and out must be non-null");
    if (rows < 1 || cols < 256 || cols % 256 != 0) return set_error(HQ_ERR_SHAPE, "need rows>=1, cols%%256==0");
    if (!aligned(W, 4) || !aligned(out, 16))
        return set_error(HQ_ERR_ALIGN, "W must be 4-byte aligned and out 16-byte aligned");
    return finish(launch_quantize(3, W, out, nullptr, rows, cols, (cudaStream_t)stream));
}

hq_status hq_quantize_i8_rows(const float *W, int8_t *Wq, float *scale, int64_t rows, int64_t cols,
                              hq_stream_t stream) {
    if (!W || !Wq || !scale) return set_error(HQ_ERR_NULL, "W, Wq and scale must be non-null");
    if (rows < 1 || rows > 0x7fffffffLL || cols < 1) return set_error(HQ_ERR_SHAPE, "need rows>=1, cols>=1");
    if (!aligned(W, 4) || !aligned(scale, 4)) return set_error(HQ_ERR_ALIGN, "W and scale must be 4-byte aligned");
    return finish(launch_quantize(2, W, Wq, scale, rows, cols, (cudaStream_t)stream));
}

hq_status hq_requant_params(const double *M, int64_t n, int32_t *mult, int32_t *shift) {
    if (!M || !mult || !shift) return set_error(HQ_ERR_NULL, "M, mult and shift must be non-null");
    for (int64_t i = 0; i < n; ++i) {
        double m = M[i];
        if (!(m > 0.0 && m < 1.0)) return set_error(HQ_ERR_UNSUPPORTED, "M[%lld] = %g not in (0,1)", (long long)i, m);
        // double m until it lies in [0.5, 1): each doubling is exact and adds one to the shift
        int s = 0;
        while (m < 0.5) { m *= 2.0; ++s; }
        long long q = llround(m * 2147483648.0);           // m * 2^31, exact before rounding
        if (q == 2147483648LL) { q = 1073741824LL; --s; }
        if (s < 0 || s > 31) return set_error(HQ_ERR_UNSUPPORTED, "M[%lld] = %g needs shift %d", (long long)i, M[i], s);
        mult[i] = (int32_t)q;
        shift[i] = s;
    }
    return finish(HQ_OK);
}

hq_status hq_requant_i32_debug(const int32_t *acc, const int32_t *mult, const int32_t *shift,
                               int8_t *y, int64_t n, int64_t rows, hq_stream_t stream) {
    if (!acc || !mult || !shift || !y) return set_error(HQ_ERR_NULL, "acc, mult, shift and y must be non-null");
    if (n < 1 || rows < 1) return set_error(HQ_ERR_SHAPE, "need n>=1, rows>=1");
    return finish(launch_requant_debug(acc, mult, shift, y, n, rows, (cudaStream_t)stream));
}

hq_status hq_selftest_wait_timeout(int64_t cycles, hq_stream_t stream) {
    if (cycles < 1 || cycles > 4000000000LL) return set_error(HQ_ERR_SHAPE, "cycles %lld not in [1, 4e9]", (long long)cycles);
    DeviceInfo *dev = nullptr;
    hq_status st = device_info(&dev);
    if (st != HQ_OK) return st;
    return finish(launch_wait_timeout_selftest(dev->fault, cycles, (cudaStream_t)stream));
}

hq_status hq_device_fault(uint32_t *fault) {
    if (!fault) return set_error(HQ_ERR_NULL, "fault must be non-null");
    DeviceInfo *dev = nullptr;
    hq_status st = device_info(&dev);
    if (st != HQ_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    uint32_t v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, dev->fault, sizeof(v), cudaMemcpyDeviceToHost);
    const uint32_t zero = 0;
    if (e == cudaSuccess) e = cudaMemcpy(dev->fault, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "reading the fault word: %s", cudaGetErrorString(e));
    *fault = v;
    if (v) return set_error(HQ_ERR_DEVICE, "device fault word 0x%x (flags 0x%x, CTA %u, %s)", v, v & 0xffu,
                            v >> 9, (v & 0x100u) ? "consumer" : "producer");
    return finish(HQ_OK);
}

}  // extern "C"
