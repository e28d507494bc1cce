// Paged decode instances for K format K_INT8_TOK (all V formats, head_dim
// 64 and 128, packed and wide GQA layouts).
#include "decode_launch.cuh"

namespace kvq {
template cudaError_t plan_decode_kf<K_INT8_TOK>(int, int, int, int, int, bool, DecodePlan *);
template cudaError_t launch_decode_kf<K_INT8_TOK>(int, int, const DecodeArgs &, const DecodePlan &,
                                               const DecodeMaps &, cudaStream_t);
}  // namespace kvq
