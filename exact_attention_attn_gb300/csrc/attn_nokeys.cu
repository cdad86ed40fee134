// Problems with no keys (Nkv == 0): every query row sees nothing, so its
// output row is 0 and its LSE is -inf (the reading the library takes for a
// row with no visible key).  One grid-stride pass of 16-byte stores over O
// and 4-byte stores over LSE.
#include <math.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) attn_nokeys_kernel(Problem p) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Nq;
  const int64_t vecs = rows * (p.D / 8);  // 8 bf16 per 16-byte store
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  uint4 *o = reinterpret_cast<uint4 *>(p.o);
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < vecs; i += stride) o[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t r = (int64_t)blockIdx.x * kThreads + threadIdx.x; r < rows; r += stride) p.lse[r] = -INFINITY;
}

}  // namespace

cudaError_t launch_nokeys(const Problem &p, int sm_count, cudaStream_t stream) {
  const int64_t vecs = (int64_t)p.B * p.Hq * p.Nq * (p.D / 8);
  int64_t blocks = (vecs + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)(sm_count > 0 ? sm_count : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  attn_nokeys_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
