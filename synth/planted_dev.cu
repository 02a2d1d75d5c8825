// CUDA twin of synth/planted.py: fills Q, K or V (bf16 bits) on the device with
// the same planted-structure values, bit for bit.  Every step is integer
// arithmetic or a single IEEE fp32 operation with explicit round-to-nearest
// (__fadd_rn / __fmul_rn), matching numpy's float32 arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

struct FillArgs {
  uint16_t* out;
  uint64_t key;      // stream key of (seed, tensor)
  int tensor;        // 1 = q, 2 = k, 3 = v
  int B, H, S, D;    // output layout [B][H][S][D]
  int G, Hkv;        // query heads per kv head, kv heads
  int Sq, Skv;
  int window, sink, rblock, nrb, nw;
  int decode;        // decode workload (exact recent window on keys, no segment directions)
  const float* tu;   // [Hkv][D]      a*u (q) or b*u (k)
  const float* tv;   // [Hkv][nw][D]  a*v_t (q) or b*v_t (k)
  const uint8_t* rblk;  // [B][Hkv][nrb]
};

__global__ void fill_kernel(FillArgs a) {
  const long long total = static_cast<long long>(a.B) * a.H * a.S * a.D;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    int acc = 0;
    const uint64_t base = a.key + 3ull * static_cast<uint64_t>(e);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const uint64_t h = splitmix64(base + j);
      acc += static_cast<int>(h & 0xFFFF) + static_cast<int>((h >> 16) & 0xFFFF) +
             static_cast<int>((h >> 32) & 0xFFFF) + static_cast<int>((h >> 48) & 0xFFFF);
    }
    float x = __fmul_rn(static_cast<float>(acc - 6 * 65535), 1.0f / 65536.0f);
    const int d = static_cast<int>(e % a.D);
    const long long row = e / a.D;
    const int s = static_cast<int>(row % a.S);
    const long long bh = row / a.S;
    const int h = static_cast<int>(bh % a.H);
    const int b = static_cast<int>(bh / a.H);
    const bool seg_dirs = !a.decode && a.window > 0;
    if (a.tensor == 1) {
      const int hk = h / a.G;
      x = __fadd_rn(x, a.tu[hk * a.D + d]);
      if (seg_dirs) {
        const int seg = (s + (a.Skv - a.Sq)) / a.window;
        x = __fadd_rn(x, a.tv[(static_cast<long long>(hk) * a.nw + seg) * a.D + d]);
        if (seg >= 1) x = __fadd_rn(x, a.tv[(static_cast<long long>(hk) * a.nw + seg - 1) * a.D + d]);
      }
    } else if (a.tensor == 2) {
      bool planted = s < a.sink ||
                     a.rblk[(static_cast<long long>(b) * a.Hkv + h) * a.nrb + s / a.rblock] != 0;
      if (a.decode && a.window > 0 && s >= a.Skv - a.window) planted = true;
      if (planted) x = __fadd_rn(x, a.tu[h * a.D + d]);
      if (seg_dirs)
        x = __fadd_rn(x, a.tv[(static_cast<long long>(h) * a.nw + s / a.window) * a.D + d]);
    }
    const uint32_t bits = __float_as_uint(x);
    a.out[e] = static_cast<uint16_t>((bits + 0x7FFFu + ((bits >> 16) & 1u)) >> 16);
  }
}

}  // namespace

extern "C" int planted_fill(uint16_t* out, unsigned long long key, int tensor, int B, int H, int S,
                            int D, int G, int Hkv, int Sq, int Skv, int window, int sink,
                            int rblock, int nrb, int nw, int decode, const float* tu,
                            const float* tv, const uint8_t* rblk, void* stream) {
  FillArgs a{out, key, tensor, B, H, S, D, G, Hkv, Sq, Skv, window, sink, rblock, nrb, nw, decode,
             tu, tv, rblk};
  fill_kernel<<<148 * 16, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return static_cast<int>(cudaGetLastError());
}
