// filler.cu -- test helper: keeps SMs busy for a bounded time, so that a
// kernel launched beside it finds only a few SMs free.
//
// Each block takes `smem_bytes` of shared memory (enough that no CTA of the
// GEMM fits on the same SM) and spins on the global timer until `ns`
// nanoseconds have passed since it started; it waits for nothing else.
// Test infrastructure only, built by the tests that use it.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void hold_sm(uint64_t ns, int* done) {
    extern __shared__ uint8_t smem[];
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    if (threadIdx.x == 0) smem[0] = 1;
    while (true) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 >= ns) break;
        __nanosleep(1000);
    }
    if (threadIdx.x == 0) atomicAdd(done, 1);
}

extern "C" int filler_launch(int blocks, int smem_bytes, unsigned long long ns, int* done, void* stream) {
    cudaError_t e = cudaFuncSetAttribute(hold_sm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    hold_sm<<<blocks, 32, smem_bytes, static_cast<cudaStream_t>(stream)>>>(ns, done);
    return static_cast<int>(cudaGetLastError());
}
