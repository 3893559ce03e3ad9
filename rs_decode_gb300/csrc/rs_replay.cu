// Replay launch entry: dispatch on the layer family and slab shape, the small
// 64 x 64 slab shapes of both families, and the host helpers of the
// column-split pipeline (tensor-map encoding, device limits).
//
// Two replay pipelines serve the two families (both persistent and
// warp-specialised, both streaming the checkpoint with bulk copies into a
// shared-memory ring):
//   * Mamba-2 (rs::rows, up to 4 drafts): the CTA's consumer warps split the
//     key rows of each staged slab and combine their partial dots through
//     shared memory; the per-unit operands are staged by the consumers
//     themselves.
//   * Gated DeltaNet, and Mamba-2 rounds of 5..8 drafts (rs::cols): each
//     consumer warp owns value columns and reduces with shuffles alone (the
//     recurrence over drafts that gives u is then warp-local), and prep warps
//     build each unit's context one unit ahead of the consumers.
#include <mutex>

#include "rs_replay_cols.cuh"
#include "rs_replay_rows.cuh"

namespace rs {
namespace cols {

namespace {

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no
// link-time dependency on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

DeviceLimits g_limits[kMaxDevices];
bool g_limits_ok[kMaxDevices];
std::mutex g_limits_mu;

}  // namespace

bool encode_slab_map(CUtensorMap *map, const void *base, bool bf16, int P, int N, long long slabs, bool col_blocks) {
    const EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t esz = bf16 ? 2 : 4, cb = 128 / esz;
    if ((P * esz) % 128 != 0 || N > 256 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
    const cuuint64_t dims[4] = {cb, (cuuint64_t)P / cb, (cuuint64_t)N, (cuuint64_t)slabs};
    const cuuint64_t strides[3] = {128, (cuuint64_t)P * esz, (cuuint64_t)N * P * esz};  // bytes, dims 1..3
    const cuuint64_t lines = (cuuint64_t)P / cb;  // 128-byte lines per row
    if (N % lines != 0 || N / lines > 256) return false;
    // one box = one row block: N / lines whole rows, i.e. N x 128 bytes; or
    // (col_blocks) one column block: the same 128-byte line of all N rows
    const cuuint32_t box[4] = {(cuuint32_t)cb, col_blocks ? 1u : (cuuint32_t)lines,
                               col_blocks ? (cuuint32_t)N : (cuuint32_t)(N / lines), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t device_limits(DeviceLimits &d) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_limits_mu);
    if (!g_limits_ok[dev]) {
        DeviceLimits l;
        if ((e = cudaDeviceGetAttribute(&l.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&l.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&l.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&l.reserved_per_block, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
            cudaSuccess)
            return e;
        g_limits[dev] = l;
        g_limits_ok[dev] = true;
    }
    d = g_limits[dev];
    return cudaSuccess;
}

}  // namespace cols

cudaError_t replay_launch_64x64(const ReplayParams &p, int kind, cudaStream_t s) {
    if (kind == RS_MAMBA2) {
        const int T = p.mode == MODE_VERIFY ? p.T : 1;
        if (T > 4) return cols::launch_pipe<cols::RCfg<RS_MAMBA2, 64, 64, 8>>(p, s);
        if (T > 1) return rows::launch_shape<RS_MAMBA2, 64, 64, 128, 4, 1, 2, 1>(p, s);
        return rows::launch_shape<RS_MAMBA2, 64, 64, 128, 1, 1, 2, 1>(p, s);
    }
    if (kind == RS_KDA) return cols::dispatch_shape<RS_KDA, 64, 64>(p, s);
    return cols::dispatch_shape<RS_GDN, 64, 64>(p, s);
}

cudaError_t replay_launch(const ReplayParams &p, int kind, int P, int N, cudaStream_t s) {
    if (replay_direct_applies(p, kind, P, N)) return replay_direct_launch(p, s);
    if (kind == RS_MAMBA2 && P == 64 && N == 128) return replay_launch_m2_64x128(p, s);
    if (kind == RS_GDN && P == 128 && N == 128) return replay_launch_gdn_128x128(p, s);
    if (kind == RS_KDA && P == 128 && N == 128) return replay_launch_kda_128x128(p, s);
    if (P == 64 && N == 64) return replay_launch_64x64(p, kind, s);
    return cudaErrorInvalidValue;
}

bool replay_shape_supported(int kind, int P, int N) {
    if (kind == RS_MAMBA2) return P == 64 && (N == 128 || N == 64);
    return (P == 128 && N == 128) || (P == 64 && N == 64);
}

}  // namespace rs
