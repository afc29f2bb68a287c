// gdn_decode_x.cu -- the decode-step kernels for the other head shapes: key and value head
// sizes that differ (dk = 128 / dv = 64 and dk = 64 / dv = 128), and square heads split along
// dv over a cluster of two CTAs (GDN_SPLIT_DV: dk == dv in {64, 128}). Same kernel as
// gdn_decode.cu (gdn_decode_kernel.cuh), separate translation unit so the two compile in
// parallel.
#include "gdn_decode_kernel.cuh"
#include "gdn_tmap.h"

namespace gdn {
namespace shaped {

cudaError_t encode_state_map(CUtensorMap* map, const float* pool, size_t rows, int DV, int box_cols, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(DV), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(DV) * 4u};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pool, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace shaped

size_t decode_smem_bytes_x(int mode, int dk, int dv, int ns, int C, int klog_bytes, int ulog_bytes) {
  return shaped::decode_layout(mode, dk, dv / ns, C, klog_bytes, ulog_bytes).total;
}

cudaError_t launch_decode_x(int mode, const DecodeParams& p, cudaStream_t stream) {
  using namespace shaped;
  const int ns = (p.flags & GDN_SPLIT_DV) ? 2 : 1;
  if (ns == 1) {
    if (p.D == 128 && p.DV == 64) return launch_decode_shape<128, 64, 1>(mode, p, stream);
    if (p.D == 64 && p.DV == 128) return launch_decode_shape<64, 128, 1>(mode, p, stream);
  } else if (ns == 2 && p.D == p.DV) {
    if (p.D == 128) return launch_decode_shape<128, 128, 2>(mode, p, stream);
    if (p.D == 64) return launch_decode_shape<64, 64, 2>(mode, p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gdn
