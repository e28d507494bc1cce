// Paged decode instances for K format K_INT2_CHAN (all V formats, head_dim
// 128, packed and wide GQA layouts).
#include "decode_launch.cuh"

namespace kvq {
template cudaError_t plan_decode_kf<K_INT2_CHAN>(int, int, int, int, int, bool, DecodePlan *);
template cudaError_t launch_decode_kf<K_INT2_CHAN>(int, int, const DecodeArgs &, const DecodePlan &,
                                               const DecodeMaps &, cudaStream_t);
}  // namespace kvq
