// Tensor-core decode-kernel instantiations for one K/V kind pair and one
// scale type (a translation unit of its own, so they compile in parallel).
#include "kvq_decode_tc.cuh"

namespace kvq {
kvq_status launch_tc_s4s4_f16(const TcArgs& t, int hd, int nt, int ng, const TcLaunchCfg& lc) {
  return launch_tc_pt<KVQ_SYM_INT4, KVQ_SYM_INT4, KVQ_F16>(t, hd, nt, ng, lc);
}
}  // namespace kvq
