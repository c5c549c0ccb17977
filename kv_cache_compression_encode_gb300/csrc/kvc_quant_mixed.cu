// kvc_quant_mixed.cu -- format-v2 instantiations of the quantize / dequantize
// kernels with per-(layer, head) code widths ("KVServe: Service-Aware KV Cache
// Compression for Communication-Efficient Disaggregated LLM Serving", §5.1,
// layer- and head-wise mixed precision; "Beyond Compression Ratio: High-Throughput
// KV Compression for Disaggregated LLM Serving", §4.1, head-importance-aware
// mixed precision kept by the fused kernel), with or without the token delta.
// A key tile takes its (layer, head)'s width per tile; the value rows run in
// (layer, head, token) order so that a warp's rows share one width.
#include "kvc_quant_kernels.cuh"

namespace kvc {

int launch_quant_mixed(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, bool enc, int sm, int cap,
                       void *st, const char **name) {
  return p.delta ? dispatch_v<0, true, true>(p, maps, *widths, enc, sm, cap, st, name)
                 : dispatch_v<0, false, true>(p, maps, *widths, enc, sm, cap, st, name);
}

}  // namespace kvc
