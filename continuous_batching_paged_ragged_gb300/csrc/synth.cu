// libpkv_synth: device-side twin of the seeded input generator (synth.py).  Input generation only --
// no attention, append or scheduling arithmetic.  Philox4x32-10 as published by Salmon, Moraes, Dror
// and Shaw ("Parallel random numbers: as easy as 1, 2, 3", SC 2011), written here from that definition;
// each value is an Irwin-Hall sum of four 16-bit uniforms, centred, scaled by float32(sqrt(3)/65536)
// in one IEEE multiply and rounded to fp16 (nearest-even), so it matches the host generator bit for bit.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
    const uint32_t n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
    const uint32_t n3 = (uint32_t)p0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

__device__ __forceinline__ __half irwin_hall(uint32_t wa, uint32_t wb, float scale) {
  const int32_t s = (int32_t)(wa & 0xFFFFu) + (int32_t)(wa >> 16) + (int32_t)(wb & 0xFFFFu) + (int32_t)(wb >> 16) -
                    131070;
  return __float2half_rn(__fmul_rn(__int2float_rn(s), scale));
}

// One thread per pair of elements of one token's [heads][dim] row.
__global__ void fill_kernel(int kind, uint64_t seed, int layer, const int64_t* __restrict__ req,
                            const int64_t* __restrict__ pos, int64_t num_tokens, int pairs_per_token, float scale,
                            __half2* __restrict__ out) {
  const int64_t total = num_tokens * pairs_per_token;
  const uint32_t k0 = (uint32_t)seed;
  const uint32_t k1 = ((uint32_t)(kind & 0xFF) << 24) | ((uint32_t)layer & 0xFFFFFFu);
  const uint32_t c3 = (uint32_t)(seed >> 32);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / pairs_per_token;
    const uint32_t pair = (uint32_t)(i - t * pairs_per_token);
    uint32_t c[4] = {pair, (uint32_t)pos[t], (uint32_t)req[t], c3};
    philox4x32_10(c, k0, k1);
    out[i] = __halves2half2(irwin_hall(c[0], c[1], scale), irwin_hall(c[2], c[3], scale));
  }
}

}  // namespace

// kind 1 = q, 2 = k, 3 = v; out: fp16 [num_tokens][heads][head_dim] (device).  Returns a cudaError_t.
extern "C" int pkv_synth_fill(int kind, uint64_t seed, int layer, const int64_t* req_ids, const int64_t* positions,
                              int64_t num_tokens, int heads, int head_dim, void* out, void* stream) {
  if (num_tokens <= 0) return 0;
  const int pairs = heads * head_dim / 2;
  const float scale = 0x1.bb67aep-16f;  // float32(sqrt(3) / 65536), bit pattern 0x37ddb3d7 as on the host side
  const int64_t total = num_tokens * pairs;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(kind, seed, layer, req_ids, positions, num_tokens,
                                                                   pairs, scale, static_cast<__half2*>(out));
  return (int)cudaGetLastError();
}
