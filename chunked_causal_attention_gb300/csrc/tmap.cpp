// Host helpers of the tcgen05 kernels: TMA tensor maps and the SM count.
#include <cudaTypedefs.h>

#include "attn_internal.h"

namespace attn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

}  // namespace

// Rank-4 map of a [B, T, H, D]-strided tensor (axes 1..3 sorted by stride),
// box = box_cols elements of the head dim x box_rows tokens, 128-byte swizzle.
static bool make_map4(CUtensorMap* m, const void* base, const Geom& g, TcMaps& mp, CUtensorMapDataType dt,
                      int elem_bytes, int box_cols, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    struct Ax {
        int64_t stride, dim;
        int which;
    } ax[3] = {{g.st, g.T, 0}, {g.sh, g.H, 1}, {g.sb, g.B, 2}};
    for (int i = 0; i < 3; ++i)
        for (int j = i + 1; j < 3; ++j)
            if (ax[j].stride < ax[i].stride) {
                Ax t = ax[i];
                ax[i] = ax[j];
                ax[j] = t;
            }
    cuuint64_t dims[4] = {(cuuint64_t)g.D, 0, 0, 0};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {(cuuint32_t)box_cols, 1, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    for (int i = 0; i < 3; ++i) {
        dims[i + 1] = (cuuint64_t)ax[i].dim;
        strides[i] = (cuuint64_t)ax[i].stride * (cuuint64_t)elem_bytes;
        if (ax[i].which == 0) {
            box[i + 1] = (cuuint32_t)box_rows;
            mp.pos_t = i + 1;
        } else if (ax[i].which == 1) {
            mp.pos_h = i + 1;
        } else {
            mp.pos_b = i + 1;
        }
    }
    CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tile_map(CUtensorMap* m, const void* base, const Geom& g, TcMaps& mp, int box_rows) {
    return make_map4(m, base, g, mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, box_rows);
}

bool make_kv_acc_map(CUtensorMap* m, float* acc, const Geom& gkv, TcMaps& mp) {
    return make_map4(m, acc, gkv, mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 32, 128);
}

bool make_dq_acc_map(CUtensorMap* m, float* dq_acc, const Geom& g, int32_t rows) {
    auto enc = encode_fn();
    if (!enc || rows <= 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)g.D, (cuuint64_t)rows, (cuuint64_t)g.B * (cuuint64_t)g.H};
    cuuint64_t strides[2] = {(cuuint64_t)g.D * 4, (cuuint64_t)rows * g.D * 4};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dq_acc, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int device_sm_count() {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) return 152;
    return c;
}

}  // namespace attn
