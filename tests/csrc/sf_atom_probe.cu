// Test-only probe of the tensor-memory placement of one 512-byte scale atom.
//
// The block-scaled MMA reads its scale factors from tensor memory.  The hardware's own way to
// put a 128x4 scale atom there is tcgen05.cp with the 32x128b.warpx4 shape: shared-memory row i
// (16 bytes) of the atom lands in lane i of every 32-lane quarter, as four 32-bit columns.  The
// GEMM kernels do not issue that copy (it would occupy the tensor pipe); their scale warps write
// the same placement with tcgen05.st.  This probe issues the hardware copy of an atom of known
// bytes and reads all 128 lanes x 4 columns back with tcgen05.ld, so that a test can compare
// the hardware's placement with the one the scale warps write.  One CTA of 128 threads; every
// wait is bounded (a wait that runs out sets *status and the probe skips the read-back).
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace {

__device__ __forceinline__ void tmem_ld_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}

__global__ void __launch_bounds__(128, 1) sf_atom_probe_kernel(const uint32_t* atom, uint32_t* out, unsigned* status) {
  __shared__ __align__(1024) uint32_t atom_s[128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  atom_s[t] = atom[t];
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the copy reads through the async proxy
  if (t == 0) {
    bsg::mbar_init(bsg::smem_u32(&bar), 1);
    bsg::fence_mbar_init();
  }
  if (warp == 0) {
    bsg::tmem_alloc(bsg::smem_u32(&tmem_slot), 32);
    bsg::tmem_relinquish();
  }
  bsg::tc_fence_before();
  __syncthreads();
  bsg::tc_fence_after();
  const uint32_t base = tmem_slot;
  if (t == 0) {
    bsg::tc_cp_sf_atom(base, bsg::sdesc_sf_atom(bsg::smem_u32(atom_s)));
    bsg::tc_commit(bsg::smem_u32(&bar));
  }
  bool done = bsg::mbar_try_wait(bsg::smem_u32(&bar), 0);
  const uint64_t t0 = bsg::globaltimer_ns();
  while (!done && bsg::globaltimer_ns() - t0 < 100000000ull) done = bsg::mbar_try_wait(bsg::smem_u32(&bar), 0);
  if (!done) atomicOr(status, 1u);
  const bool all_done = __all_sync(0xffffffffu, done);
  bsg::tc_fence_after();
  if (all_done) {
    uint32_t r[4];
    tmem_ld_x4(base + (static_cast<uint32_t>(warp * 32) << 16), r);
    bsg::tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 4; ++k) out[(warp * 32 + lane) * 4 + k] = r[k];
  }
  bsg::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    bsg::tc_fence_after();
    bsg::tmem_dealloc(base, 32);
  }
}

}  // namespace

// atom: 512 bytes (device, 16-byte aligned); out: 128 lanes x 4 words (device); status: one
// device word, OR-ed with 1 if the copy's completion was not seen within 100 ms.
extern "C" __attribute__((visibility("default"))) int sf_atom_probe(const void* atom, void* out, void* status,
                                                                    void* stream) {
  sf_atom_probe_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint32_t*>(atom), static_cast<uint32_t*>(out), static_cast<unsigned*>(status));
  return static_cast<int>(cudaGetLastError());
}
