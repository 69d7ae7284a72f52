// Tensor-core decode-kernel instantiations for unquantised f16 K and V (no
// scales; a translation unit of its own, so it compiles in parallel).
#include "kvq_decode_tc.cuh"

namespace kvq {
kvq_status launch_tc_h16(const TcArgs& t, int hd, int nt, int ng, const TcLaunchCfg& lc) {
  return launch_tc_pt<KVQ_F16_KV, KVQ_F16_KV, KVQ_F32>(t, hd, nt, ng, lc);
}
}  // namespace kvq
