// kvc_quant_delta.cu -- format-v2 instantiations of the quantize / dequantize
// kernels with the token-delta transformer ("KVServe: Service-Aware KV Cache
// Compression for Communication-Efficient Disaggregated LLM Serving", §5.1, the
// Delta transformer: each 128-token block's first row is the anchor that the
// other rows are coded against) and one code width per tensor.
#include "kvc_quant_kernels.cuh"

namespace kvc {

int launch_quant_delta(const QuantParams &p, const TmaMaps *maps, bool enc, int sm, int cap, void *st,
                       const char **name) {
  const NoWidths W = {0u};
  switch (p.bits) {
    case 2: return dispatch_v<2, true, false>(p, maps, W, enc, sm, cap, st, name);
    case 3: return dispatch_v<3, true, false>(p, maps, W, enc, sm, cap, st, name);
    case 4: return dispatch_v<4, true, false>(p, maps, W, enc, sm, cap, st, name);
    default: return dispatch_v<8, true, false>(p, maps, W, enc, sm, cap, st, name);
  }
}

}  // namespace kvc
