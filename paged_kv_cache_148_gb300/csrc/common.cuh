// Device helpers shared by the sm_103a kernels of libpagedkv.so: error flag,
// bf16 unpacking, mbarrier waits with a bound, bulk async copies (TMA engine)
// and a few PTX wrappers.  Everything is inline PTX or plain CUDA C++.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

#define PA_DEVICE __device__ __forceinline__

namespace pa {

// First device-side error wins; later ones are dropped.  Never traps.
PA_DEVICE void set_error(int32_t* d_err, int32_t code) {
    if (d_err != nullptr) atomicCAS(d_err, 0, code);
}

// bf16 pair packed in a 32-bit word -> two floats (bf16 is the top half of an
// IEEE binary32, so this is exact).
PA_DEVICE float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
PA_DEVICE float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x with the hardware approximation (MUFU.EX2); ex2(-inf) = +0.
PA_DEVICE float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

PA_DEVICE uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

PA_DEVICE uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream is finishing;
// griddep_wait() blocks until the predecessor grid has completed and its
// memory is visible (a no-op for an ordinary launch).  griddep_launch()
// lets the next kernel in the stream start launching.
PA_DEVICE void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
PA_DEVICE void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------- mbarrier
PA_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

PA_DEVICE void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

PA_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

PA_DEVICE void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

PA_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most ~timeout_ns.
// Returns false (and records PA_ERR_TIMEOUT) if the wait ran out.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legal wait

PA_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* d_err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++spins & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
            set_error(d_err, PA_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ----------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared through the TMA engine; completion is
// signalled as transaction bytes on `bar`.  src, dst and bytes must be
// multiples of 16.
PA_DEVICE void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

PA_DEVICE void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace pa
