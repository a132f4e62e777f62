// keygen.cu -- device copy of the synthetic key generator in workloads/__init__.py.
//
// Produces, bit for bit, the fp16 keys the host generator produces, so that
// large workloads can be drawn directly in device memory. Every fp64 step is
// one IEEE operation in the host's order (explicit _rn intrinsics, no fused
// multiply-add); the quantile table and the cos/sin tables come from the host.
// Input synthesis only: nothing of the eviction method is computed here.
#include <cuda_fp16.h>
#include <cstdint>

namespace {

__device__ __forceinline__ uint64_t sm64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

constexpr uint64_t TAG_KEYS = 0x4B45595F47454E31ull;
constexpr uint64_t TAG_RISER = 0x5249534552000000ull;
constexpr uint64_t RISER_THRESH = 450359962737049ull;  // int(0.05 * 2^53)
constexpr int64_t RISER_WINDOW = 1024;

struct GenArgs {
  uint16_t* out;
  const double* ninv;   // [65536]
  const double* cos_t;  // [n_pos_table, D/2], row p
  const double* sin_t;
  const double* unit;   // [D] (late riser only)
  int B, L, H, D;
  int64_t p0, count;
  int64_t sb, sl, sh, sp;  // element strides of out for b, l, h, (p - p0)
  uint64_t key_seed;
  int late_riser;
};

__device__ __forceinline__ double draw(const GenArgs& a, uint64_t hr, int d) {
  uint64_t he = sm64(hr ^ (uint64_t)d);
  return a.ninv[he >> 48];
}

__global__ void keygen_kernel(GenArgs a) {
  const int half = a.D / 2;
  const int64_t rows = (int64_t)a.B * a.L * a.H * a.count;
  const int64_t total = rows * half;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(t % half);
    int64_t r = t / half;
    const int64_t pp = r % a.count; r /= a.count;
    const int h = (int)(r % a.H); r /= a.H;
    const int l = (int)(r % a.L);
    const int b = (int)(r / a.L);
    const int64_t p = a.p0 + pp;
    uint64_t hr = sm64(a.key_seed ^ TAG_KEYS);
    hr = sm64(hr ^ (uint64_t)b);
    hr = sm64(hr ^ (uint64_t)l);
    hr = sm64(hr ^ (uint64_t)h);
    hr = sm64(hr ^ (uint64_t)p);
    double va = draw(a, hr, i);
    double vb = draw(a, hr, i + half);
    if (a.late_riser) {
      const double ua = a.unit[i], ub = a.unit[i + half];
      const bool riser = ((sm64(hr ^ TAG_RISER) >> 11) < RISER_THRESH) && (p < RISER_WINDOW);
      if (riser) {
        va = __dadd_rn(__dmul_rn(0.3, va), __dmul_rn(3.0, ua));
        vb = __dadd_rn(__dmul_rn(0.3, vb), __dmul_rn(3.0, ub));
      } else {
        const double alpha = __ddiv_rn(__dmul_rn(3.0, (double)p), 4095.0);
        va = __dadd_rn(va, __dmul_rn(alpha, ua));
        vb = __dadd_rn(vb, __dmul_rn(alpha, ub));
      }
    }
    const double c = a.cos_t[p * half + i], s = a.sin_t[p * half + i];
    const double x = __dsub_rn(__dmul_rn(va, c), __dmul_rn(vb, s));
    const double y = __dadd_rn(__dmul_rn(va, s), __dmul_rn(vb, c));
    uint16_t* o = a.out + b * a.sb + l * a.sl + h * a.sh + pp * a.sp;
    o[i] = __half_as_ushort(__double2half(x));
    o[i + half] = __half_as_ushort(__double2half(y));
  }
}

}  // namespace

extern "C" int keygen_fill(uint16_t* out, const double* ninv, const double* cos_t,
                           const double* sin_t, const double* unit, int B, int L, int H, int D,
                           int64_t p0, int64_t count, int64_t sb, int64_t sl, int64_t sh,
                           int64_t sp, uint64_t key_seed, int late_riser, void* stream) {
  GenArgs a{out, ninv, cos_t, sin_t, unit, B, L, H, D, p0, count, sb, sl, sh, sp, key_seed,
            late_riser};
  const int64_t total = (int64_t)B * L * H * count * (D / 2);
  if (total <= 0) return 0;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  keygen_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
  return (int)cudaGetLastError();
}
