// Decode-attention kernels instantiated for one (query dtype, cache dtype) pair;
// one translation unit per pair so the library builds in parallel.
#include "pkv_decode_impl.cuh"

namespace pkv {
namespace decode {
int dispatch_e4m3(const Args& a) { return dispatch<__nv_bfloat16, uint8_t>(a); }
}  // namespace decode
}  // namespace pkv
