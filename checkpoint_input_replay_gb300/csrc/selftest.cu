// rs_selftest_wait_timeout: exercises, on the GPU and without any fault, the
// bounded mbarrier wait that every hot-path kernel uses.  One thread waits on
// an mbarrier whose phase nothing completes; mbar_wait_bounded gives up after
// the limit (or 2^22 polls) exactly as it would inside a kernel whose producer
// stopped, and the outcome is written to a device word that the host reads.
#include "common.cuh"

namespace {

static __device__ int g_selftest_code;

__global__ void wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) rs::mbar_init(&bar, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: its first phase never completes
    const bool seen = rs::mbar_wait_bounded(&bar, 0, limit_ns);
    g_selftest_code = seen ? rs::DEVERR_NONE : rs::DEVERR_TIMEOUT;
  }
}

}  // namespace

extern "C" rs_status rs_selftest_wait_timeout(int32_t limit_us, int32_t* code_out, rs_stream stream) {
  if (!code_out) return RS_ERR_NULL;
  if (limit_us < 1 || limit_us > 1000000) return RS_ERR_RANGE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int minus_one = -1;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_code, &minus_one, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_us) * 1000ull);
    e = cudaGetLastError();
  }
  int code = -1;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&code, g_selftest_code, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return RS_ERR_CUDA;
  *code_out = code;
  return RS_OK;
}
