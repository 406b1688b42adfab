// Decode-attention kernels instantiated for one (query dtype, cache dtype) pair;
// one translation unit per pair so the library builds in parallel.
#include "pkv_decode_impl.cuh"

namespace pkv {
namespace decode {
int dispatch_f32(const Args& a) { return dispatch<float, float>(a); }
}  // namespace decode
}  // namespace pkv
