// ttt_internal.h -- host-side launchers shared between the C-ABI layer and the
// kernel translation units.  Not part of the public ABI (see include/ttt.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ttt {

// Problem description handed from the validated C-ABI call to a launcher.
struct LinearArgs {
    const void* Q;
    const void* K;
    const void* V;
    const float* eta;
    const float* W0;
    void* Z;
    float* W_out;
    int B, H, T, d, chunk;
    int bf16;                // 1: Q/K/V/Z are bfloat16, 0: float32
    void* W_hist = nullptr;  // optional: the state at the start of every block, [B][H][nblk][d][d],
                             // in the element type of Q (bf16: the state rounded RN-even)
    uint64_t wait_ns = 0;    // bound of the fused kernel's barrier waits (0: the default 4 s)
    // the momentum variant: M0 (nullptr: zero) and M_out [B][H][d][d] fp32
    bool momentum = false;
    const float* M0 = nullptr;
    float* M_out = nullptr;
    float beta = 0.f;
};

// Gradient of the TTT-Linear chunked scan (outer-loop training).
struct LinearBwdArgs {
    const void* Q;
    const void* K;
    const void* V;
    const float* eta;
    const void* W_hist;   // [B][H][nblk][d][d], the state at the start of every block (element type of Q)
    const void* dZ;
    const float* dW_T;    // gradient of the final state, or nullptr (zero)
    void* dQ;
    void* dK;
    void* dV;
    float* deta;
    float* dW0;
    int B, H, T, d, chunk;
    int bf16;  // 1: Q/K/V/dZ/dQ/dK/dV are bfloat16, 0: float32
};

struct MlpArgs {
    const void* Q;
    const void* K;
    const void* V;
    const float* eta;
    const float* W1_0;
    const float* W2_0;
    void* Z;
    float* W1_out;
    float* W2_out;
    int B, H, T, d, hidden, chunk;
    int bf16;
    void* W1_hist = nullptr;  // optional: the state at the start of every block, [B][H][nblk][d][hidden] and
    void* W2_hist = nullptr;  // [B][H][nblk][hidden][d], in the element type of Q
};

// Gradient of the TTT-MLP chunked scan.
struct MlpBwdArgs {
    const void* Q;
    const void* K;
    const void* V;
    const float* eta;
    const void* W1_hist;  // [B][H][nblk][d][hidden], block-start W1 (element type of Q)
    const void* W2_hist;  // [B][H][nblk][hidden][d]
    const void* dZ;
    const float* dW1_T;   // gradient of the final W1, or nullptr (zero)
    const float* dW2_T;
    void* dQ;
    void* dK;
    void* dV;
    float* deta;
    float* dW1_0;
    float* dW2_0;
    int B, H, T, d, hidden, chunk;
    int bf16;
};
bool mlp_backward_supported(int d, int hidden, int chunk);
// TTT-Linear prefill with momentum on warp-level MMAs: bf16, d = 64, chunk 16, 16 | T
// (cudaErrorNotSupported otherwise)
bool linear_momentum_mma_supported(const LinearArgs& a);
cudaError_t launch_linear_momentum_mma(const LinearArgs& a, cudaStream_t s);
cudaError_t launch_mlp_backward(const MlpBwdArgs& a, cudaStream_t s);
// warp-MMA form for bf16, d = 64, hidden = 256, chunk 16, 16 | T (cudaErrorNotSupported otherwise)
bool mlp_backward_mma_supported(const MlpBwdArgs& a);
cudaError_t launch_mlp_backward_mma(const MlpBwdArgs& a, cudaStream_t s);

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* eta;
    float* W;
    void* z;
    int B, H, d;
    int bf16;
};

struct MlpDecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* eta;
    float* W1;
    float* W2;
    void* z;
    int B, H, d, hidden;
    int bf16;
};

// Backward of the TTT-Linear scan (SIMT, fp32, one CTA per head).  bwd_supported says whether the
// block tiles of (d, chunk) fit in shared memory.
bool linear_backward_supported(int d, int chunk);
cudaError_t launch_linear_backward(const LinearBwdArgs& a, cudaStream_t s);
// Tensor-core backward for bf16, d = 64, chunk = 16, 16 | T (cudaErrorNotSupported otherwise).
cudaError_t launch_linear_backward_mma(const LinearBwdArgs& a, cudaStream_t s, int* status);

// Generic SIMT kernels: every supported shape, fp32 accumulation.
cudaError_t launch_linear_prefill_generic(const LinearArgs& a, cudaStream_t s);
cudaError_t launch_mlp_prefill_generic(const MlpArgs& a, cudaStream_t s);
size_t mlp_generic_smem_bytes(int d, int hidden, int chunk);

// TTT-Linear prefill split along the sequence (bf16, d = 64, 16 | chunk, chunk | T): nseg segments
// of seg_len tokens (a multiple of chunk; the last may be shorter); maps of every segment but the
// last, their combination into the segments' start states, then the scan of every segment.
struct SegPlan {
    int nseg;
    int seg_len;
};
bool linear_segmented_supported(const LinearArgs& a);
// force_nseg > 0 asks for that many segments (at most one per block); 0 chooses by SM count.
SegPlan linear_segment_plan(const LinearArgs& a, int force_nseg);
size_t linear_segment_workspace_bytes(const LinearArgs& a, const SegPlan& p);
cudaError_t launch_linear_prefill_segmented(const LinearArgs& a, const SegPlan& p, void* workspace, cudaStream_t s,
                                            int* status);

// Tensor-core TTT-Linear prefill (bf16, register-resident state).  Returns
// cudaErrorNotSupported when the shape is not covered, so the caller can use
// the generic kernel instead.
cudaError_t launch_linear_prefill_mma(const LinearArgs& a, cudaStream_t s, int* status);

// TTT-Linear prefill at d = 64 (bf16, 16 | chunk, chunk | T): one warp per 16-column group runs
// the recurrence and the read-out on warp-level MMAs (cudaErrorNotSupported for other shapes).
bool linear_prefill_fused_supported(const LinearArgs& a);
cudaError_t launch_linear_prefill_fused(const LinearArgs& a, cudaStream_t s, int* status);

// TTT-Linear prefill at d = 64 (bf16, 16 | chunk, chunk | T): the recurrence on
// warp-level MMAs, the read-out as per-stage tcgen05 products.
bool linear_prefill_tc_supported(const LinearArgs& a);
cudaError_t launch_linear_prefill_tc(const LinearArgs& a, cudaStream_t s, int* status);

// TTT-MLP prefill for bf16, d = 64, hidden = 256, chunk = 16 on warp-level MMAs with the state in
// registers.
bool mlp_prefill_mma_supported(const MlpArgs& a);
cudaError_t launch_mlp_prefill_mma(const MlpArgs& a, cudaStream_t s, int* status);

// Tensor-core (tcgen05) TTT-MLP prefill for bf16, d = 64, hidden = 256, chunk = 16.
bool mlp_prefill_tc_supported(const MlpArgs& a);
cudaError_t launch_mlp_prefill_tc(const MlpArgs& a, cudaStream_t s, int* status);

// TMA descriptor of a [rows][D] bf16 row-major tensor: boxes of 16 rows x 64
// columns with the 128-byte swizzle (D a multiple of 64).
cudaError_t make_tma_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, int D);
// TMA descriptor of a [heads][T][D] bf16 tensor: boxes of 16 tokens x 64 columns of one head, 128-byte
// swizzle; tokens past T read as zeros (T * D * 2 a multiple of 16 bytes).
cudaError_t make_tma_map_bf16_heads(CUtensorMap* m, const void* base, uint64_t heads, int T, int D);
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize, bytes) for `func`, once per kernel and CUDA context
cudaError_t allow_dynamic_smem(const void* func, int bytes);
// TMA descriptor of a [rows][64] fp32 row-major tensor: boxes of 64 rows x 32 columns (128 bytes),
// 128-byte swizzle (two boxes cover a 64 x 64 block).
cudaError_t make_tma_map_f32x64(CUtensorMap* m, const void* base, uint64_t rows);
// [rows][D] bf16, box box_rows x box_cols (a warp's staged output slice), swizzle 0, 64 or 128 bytes
cudaError_t make_tma_map_bf16_box(CUtensorMap* m, const void* base, uint64_t rows, int D, int box_cols,
                                  int box_rows, int swizzle_bytes);

// Device-side failure path: a bounded wait that nothing satisfies (see selftest.cu).
cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t s, int* status);

// Bandwidth-bound single-token steps.
cudaError_t launch_linear_decode(const DecodeArgs& a, cudaStream_t s, int* status);
cudaError_t launch_mlp_decode(const MlpDecodeArgs& a, cudaStream_t s);

}  // namespace ttt
