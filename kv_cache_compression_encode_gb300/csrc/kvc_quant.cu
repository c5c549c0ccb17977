// kvc_quant.cu -- launches of the fused transform + quantize + pack (encode) and
// fused reconstruction (decode) kernels of kvc_quant_kernels.cuh: the format-v1
// instantiations here, format-v2 profiles (token delta, per-(layer, head) widths)
// handed to kvc_quant_delta.cu / kvc_quant_mixed.cu.
#include "kvc_quant_kernels.cuh"

namespace kvc {

static int launch(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, bool enc, int sm, int cap,
                  void *st, uint64_t *launches, const char **name) {
  int rc;
  if (p.mixed) {
    rc = widths ? launch_quant_mixed(p, maps, widths, enc, sm, cap, st, name) : (int)cudaErrorInvalidValue;
  } else if (p.delta) {
    rc = launch_quant_delta(p, maps, enc, sm, cap, st, name);
  } else {
    const NoWidths W = {0u};
    switch (p.bits) {
      case 2: rc = dispatch_v<2, false, false>(p, maps, W, enc, sm, cap, st, name); break;
      case 3: rc = dispatch_v<3, false, false>(p, maps, W, enc, sm, cap, st, name); break;
      case 4: rc = dispatch_v<4, false, false>(p, maps, W, enc, sm, cap, st, name); break;
      default: rc = dispatch_v<8, false, false>(p, maps, W, enc, sm, cap, st, name); break;
    }
  }
  if (launches) ++*launches;
  return rc;
}

int launch_quantize(const QuantParams &p, const TmaMaps *maps, const WidthTable *widths, int sm_count, int max_per_sm,
                    void *stream, uint64_t *launches, const char **name) {
  return launch(p, maps, widths, true, sm_count, max_per_sm, stream, launches, name);
}

int launch_dequantize(const QuantParams &p, const WidthTable *widths, int sm_count, int max_per_sm, void *stream,
                      uint64_t *launches, const char **name) {
  return launch(p, nullptr, widths, false, sm_count, max_per_sm, stream, launches, name);
}

}  // namespace kvc
