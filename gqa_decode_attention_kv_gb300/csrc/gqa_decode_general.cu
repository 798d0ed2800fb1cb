// gqa_decode_general.cu -- instantiates the split-KV kernels for several new
// tokens per sequence or a sliding window (kernels in gqa_decode_kernels.cuh).
#include "gqa_decode_kernels.cuh"

namespace gqa {
namespace dec {

bool pick_general(int dtype, int kind, int d, int nw, Variant& v) {
    return pick_variant<true>(dtype, kind, d, nw, v);
}

}  // namespace dec
}  // namespace gqa
