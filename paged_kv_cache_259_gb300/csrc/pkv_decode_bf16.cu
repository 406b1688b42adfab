// Decode-attention kernels instantiated for one (query dtype, cache dtype) pair;
// one translation unit per pair so the library builds in parallel.
#include "pkv_decode_impl.cuh"

namespace pkv {
namespace decode {
int dispatch_bf16(const Args& a) { return dispatch<__nv_bfloat16, __nv_bfloat16>(a); }
}  // namespace decode
}  // namespace pkv
