// Measures the two ways a layer step can cross from one stage to the next on this GPU (the
// choice between a graph of programmatically serialised launches and one persistent launch
// with grid-wide barriers).  Built into its own library (libmono_probe.so), not the layer's.
//
//  * mono_probe_pdl_chain: one CUDA graph of n launches of a kernel whose CTAs only execute
//    griddepcontrol.launch_dependents and griddepcontrol.wait, each launch programmatically
//    serialised on the previous one -- the cost of one stage boundary of the layer's graph
//    (the layer's kernels add their own work around the same two instructions).
//  * mono_probe_grid_barrier: one cooperative launch whose CTAs cross n grid-wide barriers
//    (an arrival counter per crossing, a release arrival and an acquire spin) -- the cost of
//    one stage boundary inside a persistent kernel.  Every spin is bounded (one second): past
//    it the kernel sets an error flag and returns.
// Both time the whole sequence with CUDA events after a warm-up and return microseconds per
// boundary.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void pdl_stage_kernel() {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// counters[i] counts the CTAs past barrier i; error is set when a spin runs past its limit.
__global__ void grid_barrier_kernel(unsigned* counters, int n, int* error) {
  __shared__ int s_stop;
  const unsigned ctas = gridDim.x;
  if (threadIdx.x == 0) s_stop = 0;
  for (int i = 0; i < n; ++i) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(&counters[i], 1u);
      unsigned long long t0;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      while (ld_acquire(&counters[i]) < ctas) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > 1000000000ull) {  // one second: a peer is not coming
          atomicExch(error, 1);
          s_stop = 1;
          break;
        }
      }
    }
    __syncthreads();
    if (s_stop) return;  // (the whole CTA)
  }
}

}  // namespace

extern "C" {

// us_per_boundary: mean over n boundaries of `reps` graph replays.  Returns 0 or a CUDA error.
int mono_probe_pdl_chain(int n, int ctas, int reps, float* us_per_boundary) {
  if (n < 2 || ctas < 1 || reps < 1 || !us_per_boundary) return (int)cudaErrorInvalidValue;
  cudaStream_t s;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return (int)e;
  cudaGraph_t g = nullptr;
  cudaGraphExec_t ge = nullptr;
  cudaEvent_t t0 = nullptr, t1 = nullptr;
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pdl_stage_kernel);
  }
  const cudaError_t ec = cudaStreamEndCapture(s, &g);
  if (e == cudaSuccess) e = ec;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&ge, g, 0);
  if (e == cudaSuccess) e = cudaEventCreate(&t0);
  if (e == cudaSuccess) e = cudaEventCreate(&t1);
  for (int w = 0; w < 3 && e == cudaSuccess; ++w) e = cudaGraphLaunch(ge, s);
  if (e == cudaSuccess) e = cudaEventRecord(t0, s);
  for (int r = 0; r < reps && e == cudaSuccess; ++r) e = cudaGraphLaunch(ge, s);
  if (e == cudaSuccess) e = cudaEventRecord(t1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(t1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t0, t1);
  if (e == cudaSuccess) *us_per_boundary = ms * 1000.0f / ((float)reps * (float)n);
  if (t0) cudaEventDestroy(t0);
  if (t1) cudaEventDestroy(t1);
  if (ge) cudaGraphExecDestroy(ge);
  if (g) cudaGraphDestroy(g);
  cudaStreamDestroy(s);
  return (int)e;
}

// us_per_crossing: mean over n crossings of one cooperative launch of `ctas` CTAs (at most one
// per SM is asked for; the launch fails if they cannot all be resident).  Returns 0, a CUDA
// error, or -1 when a spin ran past its limit.
int mono_probe_grid_barrier(int n, int ctas, float* us_per_crossing) {
  if (n < 1 || ctas < 1 || !us_per_crossing) return (int)cudaErrorInvalidValue;
  unsigned* counters = nullptr;
  int* error = nullptr;
  cudaEvent_t t0 = nullptr, t1 = nullptr;
  cudaError_t e = cudaMalloc(&counters, sizeof(unsigned) * (size_t)n * 2);
  if (e == cudaSuccess) e = cudaMalloc(&error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(error, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaEventCreate(&t0);
  if (e == cudaSuccess) e = cudaEventCreate(&t1);
  float ms = 0.0f;
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {  // a warm-up pass, then timed
    unsigned* c = counters + (size_t)pass * n;
    e = cudaMemset(c, 0, sizeof(unsigned) * (size_t)n);
    void* args[] = {&c, &n, &error};
    if (e == cudaSuccess) e = cudaEventRecord(t0, 0);
    if (e == cudaSuccess)
      e = cudaLaunchCooperativeKernel((const void*)grid_barrier_kernel, dim3(ctas), dim3(128),
                                      args, 0, 0);
    if (e == cudaSuccess) e = cudaEventRecord(t1, 0);
    if (e == cudaSuccess) e = cudaEventSynchronize(t1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t0, t1);
  }
  int err = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&err, error, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) *us_per_crossing = ms * 1000.0f / (float)n;
  if (t0) cudaEventDestroy(t0);
  if (t1) cudaEventDestroy(t1);
  if (counters) cudaFree(counters);
  if (error) cudaFree(error);
  if (e != cudaSuccess) return (int)e;
  return err ? -1 : 0;
}

}  // extern "C"
