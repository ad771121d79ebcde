// Expert weights in 128 x 128-byte tiles (MOE_LAYOUT_TILES): the tensor-core
// kernels load a weight tile as one 128-row x 128-byte box per K block; in the
// row-major layout that box gathers 128 runs of 128 bytes, one per row, K
// bytes apart.  Packed, every box is 16 KB of consecutive memory, which HBM
// streams more efficiently (the weights are read once per layer call).  Within
// a tile the 16-byte chunks of row r are stored in the order the tensor cores
// read them from shared memory (128-byte swizzle: chunk c at position
// c ^ (r mod 8)), so a plain 16 KB bulk copy places a tile as the swizzling
// tensor copy would; such copies stream faster than 2-D tensor boxes.
//
//   dst[((b * KBt + kb) * 128 + r) * 128 + 16 (c ^ (r mod 8)) + j]
//       = src[(b * 128 + r) * Kbytes + kb * 128 + 16 c + j]
//
// for row block b over all groups (N % 128 == 0, so blocks never straddle
// groups), K block kb of 128 bytes, row r, 16-byte chunk c and byte j.
#include <algorithm>

#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
    pack_tiles_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int kbt,
                      int64_t total_vec) {
    // one 16-byte vector per thread and step; a tile is 128 rows x 8 vectors
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total_vec;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = v >> 10;
        const int within = (int)(v & 1023);
        const int r = within >> 3, c = within & 7;
        const int64_t b = tile / kbt;
        const int kb = (int)(tile - b * kbt);
        // destination chunk c of row r holds source chunk c ^ (r mod 8)
        dst[v] = __ldg(src + (b * 128 + r) * ((int64_t)kbt * 8) + kb * 8 + (c ^ (r & 7)));
    }
}

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_pack_expert_weights(const moe_config *cfg, int32_t groups,
                                               int32_t n_out, int32_t k_dim, const void *w,
                                               void *w_tiled, void *stream) {
    int rc = moe::check_config(cfg);
    if (rc) return rc;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (groups <= 0 || n_out <= 0 || k_dim <= 0 || !w || !w_tiled) return MOE_ERR_INVALID_ARG;
    if (n_out % 128 || k_dim % (fp8 ? 128 : 64)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!moe::aligned16(w) || !moe::aligned16(w_tiled)) return MOE_ERR_INVALID_ARG;
    const int64_t bytes = (int64_t)groups * n_out * k_dim * (fp8 ? 1 : 2);
    const char *a = static_cast<const char *>(w);
    const char *b = static_cast<const char *>(w_tiled);
    if (a < b + bytes && b < a + bytes) return MOE_ERR_INVALID_ARG;   // overlapping buffers
    const int kbt = (int)(k_dim * (fp8 ? 1 : 2) / 128);
    const int64_t total_vec = bytes / 16;
    const unsigned grid =
        (unsigned)std::min<int64_t>((total_vec + 255) / 256, (int64_t)moe::sm_count() * 16);
    moe::pack_tiles_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(w), static_cast<uint4 *>(w_tiled), kbt, total_vec);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}
