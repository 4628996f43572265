// Device helpers shared by the tensor-core kernels: bounded waits, the
// published-state flags, decay powers and the packed-bf16 feature map.
#pragma once

#include "la_internal.h"
#include "la_tc_ptx.cuh"

namespace la {
namespace tcc {

using namespace la::tc;

constexpr int FLAG_AGG = 1, FLAG_INCL = 2;
constexpr uint32_t kBf16One2 = 0x3F803F80u;    // (1, 1)
constexpr uint32_t kBf16Log2e2 = 0x3FB93FB9u;  // (log2 e, log2 e) in bf16

struct Ctx {
    volatile int *abort;  // set once any wait of the launch gave up
    int *status;          // device status word
    long long timeout;    // clock cycles per bounded wait
};

// Records the first wait that gave up: block index and an identifier (the
// barrier's shared-memory offset, or the low bits of a flag's address).
__device__ __forceinline__ void raise_timeout(const Ctx &cx, uint32_t where) {
    if (atomicCAS(cx.status, 0, (int)LA_ERR_TIMEOUT) == 0)
        atomicExch(cx.status + 1, (int)((blockIdx.x << 20) | (where & 0xFFFFFu)));
    *cx.abort = 1;
}

// Bounded mbarrier wait; passes through (returns false) once aborted.  The
// single-thread roles (TMA producer, MMA issuer) poll with test_wait, which
// never suspends, so that they react at once; warps of the multi-warp roles
// suspend between polls for at most `kSuspendNs`, so that waiting warps do
// not take issue slots from the working ones.  The abort flag lives in
// global memory, so it is read only every 64 polls; the deadline starts at
// the first of those checks.
constexpr uint32_t kSuspendNs = 64;

static __device__ __noinline__ bool wait_bar_poll(uint64_t *bar, uint32_t parity,
                                                  const Ctx &cx, bool spin) {
    long long dl = 0;
    for (int n = 1;; ++n) {
        if (spin ? mbar_test_wait(bar, parity) : mbar_try_wait_ns(bar, parity, kSuspendNs))
            return true;
        if ((n & 63) == 0) {
            if (*cx.abort) return false;
            const long long now = clock64();
            if (dl == 0) {
                dl = now + cx.timeout;
            } else if (now > dl) {
                raise_timeout(cx, smem_u32(bar));
                return false;
            }
        }
    }
}

// For warps of the multi-warp roles.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity,
                                         const Ctx &cx) {
    if (mbar_test_wait(bar, parity)) return true;
    return wait_bar_poll(bar, parity, cx, false);
}

// For the single-thread roles.
__device__ __forceinline__ bool wait_bar_spin(uint64_t *bar, uint32_t parity,
                                              const Ctx &cx) {
    if (mbar_test_wait(bar, parity)) return true;
    return wait_bar_poll(bar, parity, cx, true);
}

// A wait for the phase itself that ignores the abort flag (bounded all the
// same, far above any wait limit).  Used where the real completion matters
// whatever happened elsewhere: the item ring, whose entries all warps of a
// role must read alike (their named-barrier counts follow from the item); a
// TMA full barrier before it is armed again (one arrival per phase); and the
// drain at exit, so that no TMA load or MMA is still in flight when the CTA's
// shared memory and TMEM are released.
constexpr long long kSettleCycles = 1LL << 34;

static __device__ __noinline__ void settle_wait_poll(uint64_t *bar, uint32_t parity) {
    const long long dl = clock64() + kSettleCycles;
    while (!mbar_try_wait_ns(bar, parity, kSuspendNs) && clock64() <= dl) {
    }
}

__device__ __forceinline__ void settle_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_test_wait(bar, parity)) return;
    settle_wait_poll(bar, parity);
}

// Reads a published-state flag (acquire, device scope).
__device__ __forceinline__ int load_flag(const int *f) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}

// Bounded poll until *f >= want; returns the value seen (or `give_up` once
// aborted or timed out).
__device__ __forceinline__ int poll_flag_at_least(const int *f, int want,
                                                  int give_up, const Ctx &cx) {
    const long long dl = clock64() + cx.timeout;
    for (;;) {
        const int v = load_flag(f);
        if (v >= want) return v;
        if (*cx.abort) return give_up;
        if (clock64() > dl) {
            raise_timeout(cx, 0x80000u | ((uint32_t)(reinterpret_cast<uintptr_t>(f) >> 2) & 0x7FFFFu));
            return give_up;
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ void publish_flag(int *f, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v)
                 : "memory");
}

// g^k from log2(g) (log2(0) = -inf gives 0 for k > 0); k = 0 gives 1.
__device__ __forceinline__ float gpow(float lg, int k) {
    return k == 0 ? 1.f : exp2f(lg * (float)k);
}

__device__ __forceinline__ float head_log2g(const DecayArgs &dk, int bh) {
    if (!dk.has) return 0.f;
    return log2f(dk.g[bh % dk.H]);
}

// elu(x) + 1 on two packed bf16 values: max(x, 0) + 2^(min(x, 0) log2 e)
__device__ __forceinline__ uint32_t phi2(uint32_t x) {
    return bf2_add(bf2_max(x, 0u), bf2_ex2(bf2_mul(bf2_min(x, 0u), kBf16Log2e2)));
}

__device__ __forceinline__ uint32_t bf2_splat(float w) {
    return pack_bf16x2(w, w);
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// Offset of K-step `ks` (16 elements) in a K-major, 128-byte-swizzled tile
// made of 64-element atoms of `atom_bytes` each.
__device__ __forceinline__ uint32_t kmajor_off(int ks, uint32_t atom_bytes) {
    return (uint32_t)(ks >> 2) * atom_bytes + (uint32_t)(ks & 3) * 32u;
}

// ---------------------------------------------------------------- row transforms

// phi (bf16 pairs) over this thread's share of one row of a [128][DK]
// swizzled tile, in place (identity when `phi` is false); rows with `zero`
// set become 0.
template <int DK>
__device__ __forceinline__ void transform_row(uint8_t *tile, int row, int part,
                                              bool zero, bool phi) {
    constexpr int NCH = DK / 16;  // 16-byte chunks per thread (half a row)
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int cc = part * NCH + i;
        const uint32_t off = (cc >> 3) * 16384 + sw128_offset(row, (cc & 7) * 8);
        const uint4 x = *reinterpret_cast<const uint4 *>(tile + off);
        uint4 y = x;
        if (phi) {
            y.x = phi2(x.x);
            y.y = phi2(x.y);
            y.z = phi2(x.z);
            y.w = phi2(x.w);
        }
        if (zero) y = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(tile + off) = y;
    }
}

// Khat = w phi(K) in place (phase A weights relative to the segment end);
// w K with the identity feature map.
template <int DK>
__device__ __forceinline__ void transform_row_scaled(uint8_t *tile, int row,
                                                     int part, uint32_t w2,
                                                     bool phi) {
    constexpr int NCH = DK / 16;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int cc = part * NCH + i;
        const uint32_t off = (cc >> 3) * 16384 + sw128_offset(row, (cc & 7) * 8);
        const uint4 x = *reinterpret_cast<const uint4 *>(tile + off);
        uint4 y;
        y.x = bf2_mul(phi ? phi2(x.x) : x.x, w2);
        y.y = bf2_mul(phi ? phi2(x.y) : x.y, w2);
        y.z = bf2_mul(phi ? phi2(x.z) : x.z, w2);
        y.w = bf2_mul(phi ? phi2(x.w) : x.w, w2);
        *reinterpret_cast<uint4 *>(tile + off) = y;
    }
}

// Row `row` of a [128][DK] swizzled bf16 tile times w (this thread's half).
template <int DK>
__device__ __forceinline__ void scale_row(uint8_t *tile, int row, int part,
                                          uint32_t w2) {
    constexpr int NCH = DK / 16;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int cc = part * NCH + i;
        const uint32_t off = (cc >> 3) * 16384 + sw128_offset(row, (cc & 7) * 8);
        const uint4 x = *reinterpret_cast<const uint4 *>(tile + off);
        *reinterpret_cast<uint4 *>(tile + off) =
            make_uint4(bf2_mul(x.x, w2), bf2_mul(x.y, w2), bf2_mul(x.z, w2),
                       bf2_mul(x.w, w2));
    }
}

}  // namespace tcc
}  // namespace la
