// Tensor-core decode-kernel instantiations for the /7.5 offset-8 4-bit codec
// (shimmy4) with f32 scales (a translation unit of its own, so it compiles in
// parallel).
#include "kvq_decode_tc.cuh"

namespace kvq {
kvq_status launch_tc_o4o4_f32(const TcArgs& t, int hd, int nt, int ng, const TcLaunchCfg& lc) {
  return launch_tc_pt<KVQ_SHIMMY_INT4, KVQ_SHIMMY_INT4, KVQ_F32>(t, hd, nt, ng, lc);
}
}  // namespace kvq
