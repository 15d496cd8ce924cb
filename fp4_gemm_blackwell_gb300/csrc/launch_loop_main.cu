// Launch-overhead loop through the C ABI (the host path a C/C++ caller pays, without an FFI):
// 1000 back-to-back nvfp4_gemm calls cycling M in {1, 16, 128, 1024} x (N, K) in
// {(4096, 4096), (14336, 4096), (4096, 14336)}, BF16 output, cached plans.  Prints one JSON
// line: host enqueue time per call on a stream, wall time per call, device time per call of
// the same calls replayed from a captured CUDA graph, and host time per call of that replay.
// Then one plan of the 128 x 4096 x 4096 shape: host time per call of bsg_plan_run, and of
// bsg_plan_run_operands alternating between two buffer sets (the pointer-agnostic run, which
// checks every buffer against its allocation).  Then, as context, the per-call host path that the
// launch-overhead page profiles: bsg_gemm_noalloc, which validates, chooses the variant and
// encodes both tensor maps on every call, and the same with a driver entry-point lookup of
// cuTensorMapEncodeTiled before every call.  Operands are quantised on the device by
// bsg_quantize from a deterministic pattern.
#include <cuda_runtime.h>

#include <chrono>
#include <cstdio>
#include <vector>

#include "bsgemm.h"

namespace {

__global__ void fill_pattern(float* x, long long n, unsigned seed) {
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += 256LL * gridDim.x) {
    const unsigned h = static_cast<unsigned>(i) * 2654435761u + seed * 40503u;
    x[i] = static_cast<float>(h % 2001u) / 500.0f - 2.0f;
  }
}

struct Operand {
  void* codes = nullptr;
  void* sf = nullptr;
  float scale = 0.0f;
};

bool make_operand(int rows, int K, unsigned seed, float* xbuf, float* gs, Operand* op) {
  const long long n = static_cast<long long>(rows) * K;
  fill_pattern<<<1024, 256>>>(xbuf, n, seed);
  if (cudaMalloc(&op->codes, n / 2) != cudaSuccess) return false;
  if (cudaMalloc(&op->sf, bsg_sf_bytes(BSG_NVFP4, rows, K)) != cudaSuccess) return false;
  if (bsg_quantize(BSG_NVFP4, xbuf, rows, K, op->codes, op->sf, gs, nullptr) != BSG_OK) return false;
  if (cudaMemcpy(&op->scale, gs, sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess) return false;
  return true;
}

double now_us() {
  return std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now().time_since_epoch()).count();
}

}  // namespace

int main() {
  const int calls = 1000;
  struct Shape { int M, N, K; };
  std::vector<Shape> shapes;
  for (int m : {1, 16, 128, 1024})
    for (auto nk : {std::make_pair(4096, 4096), std::make_pair(14336, 4096), std::make_pair(4096, 14336)})
      shapes.push_back({m, nk.first, nk.second});
  float* xbuf = nullptr;
  float* gs = nullptr;
  if (cudaMalloc(&xbuf, sizeof(float) * 14336LL * 4096) != cudaSuccess || cudaMalloc(&gs, sizeof(float)) != cudaSuccess) {
    std::printf("{\"error\": \"allocation\"}\n");
    return 1;
  }
  struct Call { Operand a, b; void* d; float alpha; Shape s; };
  std::vector<Call> cl;
  unsigned seed = 1;
  for (const Shape& s : shapes) {
    Call c{};
    c.s = s;
    if (!make_operand(s.M, s.K, seed++, xbuf, gs, &c.a) || !make_operand(s.N, s.K, seed++, xbuf, gs, &c.b) ||
        cudaMalloc(&c.d, static_cast<size_t>(s.M) * s.N * 2) != cudaSuccess) {
      std::printf("{\"error\": \"operands: %s\"}\n", bsg_last_error());
      return 1;
    }
    c.alpha = c.a.scale * c.b.scale;
    cl.push_back(c);
  }
  cudaStream_t stream;
  cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking);
  auto issue = [&](int i) {
    const Call& c = cl[i % cl.size()];
    return nvfp4_gemm(c.d, c.a.codes, c.b.codes, c.a.sf, c.b.sf, nullptr, c.alpha, 0u, c.s.M, c.s.N, c.s.K,
                      BSG_OUT_BF16, reinterpret_cast<bsg_stream_t>(stream));
  };
  for (int i = 0; i < 3 * static_cast<int>(cl.size()); ++i)  // plan-cache misses, untimed
    if (issue(i) != BSG_OK) {
      std::printf("{\"error\": \"%s\"}\n", bsg_last_error());
      return 1;
    }
  cudaStreamSynchronize(stream);
  const double t0 = now_us();
  for (int i = 0; i < calls; ++i) issue(i);
  const double t1 = now_us();
  cudaStreamSynchronize(stream);
  const double t2 = now_us();
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  cudaStreamBeginCapture(stream, cudaStreamCaptureModeGlobal);
  for (int i = 0; i < calls; ++i) issue(i);
  cudaStreamEndCapture(stream, &graph);
  cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphLaunch(exec, stream);  // upload
  cudaStreamSynchronize(stream);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0, stream);
  const double g0 = now_us();
  cudaGraphLaunch(exec, stream);
  const double g1 = now_us();
  cudaEventRecord(e1, stream);
  cudaStreamSynchronize(stream);
  float ms = 0.0f;
  cudaEventElapsedTime(&ms, e0, e1);
  // one plan, two buffer sets of the 128 x 4096 x 4096 shape
  const Call* c0 = nullptr;
  for (const Call& c : cl)
    if (c.s.M == 128 && c.s.N == 4096 && c.s.K == 4096) c0 = &c;
  Operand a2, b2;
  void* d2 = nullptr;
  if (c0 == nullptr || !make_operand(128, 4096, 91, xbuf, gs, &a2) || !make_operand(4096, 4096, 92, xbuf, gs, &b2) ||
      cudaMalloc(&d2, 128 * 4096 * 2) != cudaSuccess) {
    std::printf("{\"error\": \"second operand set\"}\n");
    return 1;
  }
  bsg_desc d{};
  d.kind = BSG_NVFP4;
  d.out = BSG_OUT_BF16;
  d.M = 128;
  d.N = 4096;
  d.K = 4096;
  d.A = c0->a.codes;
  d.B = c0->b.codes;
  d.SFA = c0->a.sf;
  d.SFB = c0->b.sf;
  d.D = c0->d;
  d.alpha = c0->alpha;
  bsg_plan_t plan = nullptr;
  if (bsg_plan_create(&plan, &d) != BSG_OK) {
    std::printf("{\"error\": \"%s\"}\n", bsg_last_error());
    return 1;
  }
  bsg_operands ops[2] = {{c0->a.codes, c0->b.codes, c0->a.sf, c0->b.sf, c0->d},
                         {a2.codes, b2.codes, a2.sf, b2.sf, d2}};
  const bsg_stream_t st = reinterpret_cast<bsg_stream_t>(stream);
  for (int i = 0; i < 20; ++i) bsg_plan_run_operands(plan, &ops[i & 1], st);
  cudaStreamSynchronize(stream);
  const double r0 = now_us();
  for (int i = 0; i < calls; ++i) bsg_plan_run(plan, st);
  const double r1 = now_us();
  cudaStreamSynchronize(stream);
  const double o0 = now_us();
  int bad = 0;
  for (int i = 0; i < calls; ++i) bad += bsg_plan_run_operands(plan, &ops[i & 1], st) != BSG_OK;
  const double o1 = now_us();
  cudaStreamSynchronize(stream);
  bsg_plan_destroy(plan);
  for (int i = 0; i < 20; ++i) bad += bsg_gemm_noalloc(&d, st) != BSG_OK;  // first call finds the scratch
  cudaStreamSynchronize(stream);
  const double n0 = now_us();
  for (int i = 0; i < calls; ++i) bad += bsg_gemm_noalloc(&d, st) != BSG_OK;
  const double n1 = now_us();
  cudaStreamSynchronize(stream);
  const double x0 = now_us();
  for (int i = 0; i < calls; ++i) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    bad += bsg_gemm_noalloc(&d, st) != BSG_OK;
  }
  const double x1 = now_us();
  cudaStreamSynchronize(stream);
  const cudaError_t err = cudaGetLastError();
  const double kernel_us = ms * 1000.0 / calls;
  std::printf("{\"calls\": %d, \"shapes\": %d, \"host_us_per_call\": %.3f, \"wall_us_per_call\": %.3f, "
              "\"kernel_us_per_call\": %.3f, \"graph_host_us_per_call\": %.4f, \"host_over_kernel\": %.4f, "
              "\"plan_run_host_us\": %.3f, \"plan_run_operands_host_us\": %.3f, \"reencode_host_us\": %.3f, "
              "\"reencode_and_lookup_host_us\": %.3f, \"errors\": %d, \"cuda\": \"%s\"}\n",
              calls, static_cast<int>(cl.size()), (t1 - t0) / calls, (t2 - t0) / calls, kernel_us,
              (g1 - g0) / calls, (t1 - t0) / calls / kernel_us, (r1 - r0) / calls, (o1 - o0) / calls,
              (n1 - n0) / calls, (x1 - x0) / calls, bad, cudaGetErrorString(err));
  return err == cudaSuccess ? 0 : 1;
}
