// hq_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hq.h"

namespace hq {

// Per-device state set up once: SM count, the fault word's device address,
// and the driver's tensor-map encoder.
struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *fault = nullptr;
    float *lora_scratch = nullptr;   // static device scratch of the allocation-free QLoRA call
};

hq_status device_info(DeviceInfo **out);            // current device
void note_launch();                                 // counts each kernel launch the library makes
hq_status set_error(hq_status st, const char *fmt, ...);
void *tensor_map_encoder();                         // PFN_cuTensorMapEncodeTiled

// QLoRA adapter epilogue of a float matvec: y += scale * B u, where u = A x
// was computed by launch_lora_down earlier on the same stream.
struct MatvecExtras {
    const uint16_t *B = nullptr;    // bf16 [rows][rank]
    const float *u = nullptr;       // fp32 [n_vec][rank]
    float scale = 0.f;
    int rank = 0;                   // 0: no adapter
};

// Launchers (arguments already validated by the API layer).
hq_status launch_matvec_float_q8_0(const void *W, const float *x, float *y, int64_t rows,
                                   int64_t cols, int n_vec, const MatvecExtras *lora, cudaStream_t stream);
hq_status launch_matvec_float_q4_0(const void *W, const float *x, float *y, int64_t rows,
                                   int64_t cols, int n_vec, const MatvecExtras *lora, cudaStream_t stream);
hq_status launch_matvec_float_q4_k(const void *W, const float *x, float *y, int64_t rows,
                                   int64_t cols, int n_vec, const MatvecExtras *lora, cudaStream_t stream);
hq_status launch_lora_down(const uint16_t *A, const float *x, float *u, int rank, int64_t cols,
                           int n_vec, cudaStream_t stream);
// MoE epilogue of a grouped Q8_0 launch: 0 none; 1 SwiGLU over interleaved
// gate/up rows (y gets [n_vec][n_active][rows/2]); 2 router-weighted sum over
// the slots (y gets [n_vec][rows]).
struct MoeEpi {
    int kind = 0;
    const float *router_w = nullptr;    // [n_vec][n_active]
    int ids_ready = 0;                  // the ids do not come from the previous kernel in the stream
};
hq_status launch_moe_q8_0(const void *W_bank, const int32_t *ids, const float *x, int x_per_slot,
                          float *y, int64_t n_experts, int n_active, int64_t rows, int64_t cols,
                          int n_vec, const MoeEpi *epi, cudaStream_t stream);
hq_status launch_matvec_i8(const int8_t *W, const int8_t *x, const int32_t *mult,
                           const int32_t *shift, int8_t *y, int64_t rows, int64_t cols, int n_vec,
                           cudaStream_t stream);
hq_status launch_wait_timeout_selftest(uint32_t *fault, int64_t cycles, cudaStream_t stream);
hq_status launch_requant_debug(const int32_t *acc, const int32_t *mult, const int32_t *shift,
                               int8_t *y, int64_t n, int64_t rows, cudaStream_t stream);
hq_status launch_quantize(int fmt, const float *W, void *out, float *scale, int64_t rows,
                          int64_t cols, cudaStream_t stream);
// Test-only plan queries (no device touched): see hq_debug_plan in hq.h.
hq_status debug_plan_float_q8_0(int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs,
                                int64_t *out);
hq_status debug_plan_float_q4_0(int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs,
                                int64_t *out);
hq_status debug_plan_float_q4_k(int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs,
                                int64_t *out);
hq_status debug_plan_i8(int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs, int64_t *out);

}  // namespace hq
