// tma_host.cu -- host-side construction of the TMA tensor descriptors the
// prefill kernels stream Q, K and V through.
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "ttt_internal.h"

namespace ttt {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static cudaError_t get_encoder(EncodeTiledFn* fn) {
    static EncodeTiledFn cached = nullptr;
    if (!cached) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !p) return cudaErrorSymbolNotFound;
        cached = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = cached;
    return cudaSuccess;
}

// Encoded descriptors of this thread's recent calls, so that a serving loop over the same buffers encodes
// each once: a descriptor holds only the address and the layout, so the key (base, rows, columns, box,
// swizzle, element size) determines it.
namespace {
struct MapKey {
    const void* base;
    uint64_t rows;
    int cols, box_cols, box_rows, swizzle, elt;
    uint64_t planes;  // 0 for a 2D map, else the extent of the third dimension
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && cols == o.cols && box_cols == o.box_cols &&
               box_rows == o.box_rows && swizzle == o.swizzle && elt == o.elt && planes == o.planes;
    }
};
constexpr int kMapCache = 16;
thread_local MapKey t_keys[kMapCache];
thread_local CUtensorMap t_maps[kMapCache];
thread_local int t_used = 0, t_next = 0;

bool cached_map(const MapKey& k, CUtensorMap* m) {
    for (int i = 0; i < t_used; ++i)
        if (t_keys[i] == k) {
            *m = t_maps[i];
            return true;
        }
    return false;
}
void remember_map(const MapKey& k, const CUtensorMap& m) {
    const int i = t_used < kMapCache ? t_used++ : (t_next++ % kMapCache);
    t_keys[i] = k;
    t_maps[i] = m;
}
}  // namespace

// [rows][D] bf16 viewed as a 2D tensor; box = 16 rows x 64 columns, 128-byte swizzle.
cudaError_t make_tma_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, int D) {
    const MapKey key{base, rows, D, 64, 16, 128, 2, 0};
    if (cached_map(key, m)) return cudaSuccess;
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    remember_map(key, *m);
    return cudaSuccess;
}

// [heads][T][D] bf16 viewed as a 3D tensor; box = 16 tokens x 64 columns of one head, 128-byte swizzle.
// A box that reaches past a head's last token reads zeros there, not the next head's rows.
cudaError_t make_tma_map_bf16_heads(CUtensorMap* m, const void* base, uint64_t heads, int T, int D) {
    const MapKey key{base, uint64_t(T), D, 64, 16, 128, 2, heads};
    if (cached_map(key, m)) return cudaSuccess;
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(T), cuuint64_t(heads)};
    cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(T) * D * 2};
    cuuint32_t box[3] = {64, 16, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    remember_map(key, *m);
    return cudaSuccess;
}

// [rows][D] bf16 viewed as a 2D tensor; box = box_rows x box_cols: a slice a warp stages for a TMA store
// (box_cols * 2 bytes a multiple of 16).  swizzle_bytes: 0 (row-major in shared memory), 64 or 128 (the
// 16-byte chunks of each box row XOR bits 7.. of the shared-memory offset, as the tensor core's swizzle
// modes define; the box row is then at most that many bytes).
cudaError_t make_tma_map_bf16_box(CUtensorMap* m, const void* base, uint64_t rows, int D, int box_cols,
                                  int box_rows, int swizzle_bytes) {
    const MapKey key{base, rows, D, box_cols, box_rows, swizzle_bytes, 2, 0};
    if (cached_map(key, m)) return cudaSuccess;
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    remember_map(key, *m);
    return cudaSuccess;
}

// [rows][64] fp32 viewed as a 2D tensor; box = 64 rows x 32 columns (128 bytes), 128-byte swizzle.
cudaError_t make_tma_map_f32x64(CUtensorMap* m, const void* base, uint64_t rows) {
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {64, cuuint64_t(rows)};
    cuuint64_t strides[1] = {64 * 4};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and CUDA context (a device reset makes
// a new context, which asks again): the attribute call is a driver round trip that a serving loop would
// otherwise pay on every launch.
cudaError_t allow_dynamic_smem(const void* func, int bytes) {
    constexpr int kSlots = 128;
    static std::mutex mu;
    static struct Slot {
        const void* func;
        void* ctx;
        int bytes;
    } slots[kSlots];
    static int nslots = 0;
    static CtxGetCurrentFn get_ctx = nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!get_ctx) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !f) return cudaErrorSymbolNotFound;
        get_ctx = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)  // no context yet: let the runtime make one
        return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    for (int i = 0; i < nslots; ++i)
        if (slots[i].func == func && slots[i].ctx == static_cast<void*>(ctx) && slots[i].bytes >= bytes)
            return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
        int i = 0;
        while (i < nslots && !(slots[i].func == func && slots[i].ctx == static_cast<void*>(ctx))) ++i;
        if (i == nslots && nslots < kSlots) ++nslots;
        if (i < kSlots) slots[i] = {func, static_cast<void*>(ctx), bytes};
    }
    return e;
}

}  // namespace ttt
