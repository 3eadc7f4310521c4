// decode_d64.cu -- the decode kernel's instantiations for head_dim 64 with
// run-time head counts (groups of 1, 2, 4 and 8 query heads per KV head).
#include "decode_kernel.cuh"

namespace pkv {

int launch_decode_d64(const DecodeLaunch& c, int G) {
  switch (G) {
    case 1: return launch_decode_geo<DecGeo<64, 1, false>>(c);
    case 2: return launch_decode_geo<DecGeo<64, 2, false>>(c);
    case 4: return launch_decode_geo<DecGeo<64, 4, false>>(c);
    case 8: return launch_decode_geo<DecGeo<64, 8, false>>(c);
    default: return PKV_ERR_UNSUPPORTED;
  }
}

}  // namespace pkv
