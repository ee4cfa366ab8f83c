// The decode kernel's 8-bit cache instances (E4M3 codes, one power-of-two scale per cached row), compiled
// apart from the fp16 ones so that the two sets build in parallel.
#include "decode.cuh"

namespace pkv {

cudaError_t launch_decode_e4m3(int head_dim, int group, const DecodeParams& p, int num_sms, int64_t max_tasks,
                               cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_g<64, kKvE4M3>(group, p, num_sms, max_tasks, stream);
    case 128: return launch_decode_g<128, kKvE4M3>(group, p, num_sms, max_tasks, stream);
    case 256: return launch_decode_g<256, kKvE4M3>(group, p, num_sms, max_tasks, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
