// Shared device/host helpers of the questsparse kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/questsparse.h"

#define QS_DEVINL __device__ __forceinline__

namespace qs {

// ---------------------------------------------------------------------------
// status
// ---------------------------------------------------------------------------

// First device-side error wins; later ones are dropped.
QS_DEVINL void set_status(int32_t* st, int code) {
    if (st) atomicCAS(st, 0, code);
}

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------

enum class Dt : int { F32 = QS_F32, BF16 = QS_BF16, F16 = QS_F16, I8 = QS_I8 };

template <Dt T> struct DtInfo;
template <> struct DtInfo<Dt::F32> { static constexpr int bytes = 4; };
template <> struct DtInfo<Dt::BF16> { static constexpr int bytes = 2; };
template <> struct DtInfo<Dt::F16> { static constexpr int bytes = 2; };
template <> struct DtInfo<Dt::I8> { static constexpr int bytes = 1; };

// bf16 pair in one 32-bit word -> two floats (exact).
QS_DEVINL float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
QS_DEVINL float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

QS_DEVINL float f16lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
QS_DEVINL float f16hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Two consecutive elements held in word w (16-bit dtypes) as floats.
template <Dt T> QS_DEVINL float2 pair_to_float2(uint32_t w);
template <> QS_DEVINL float2 pair_to_float2<Dt::BF16>(uint32_t w) {
    return make_float2(bf16lo(w), bf16hi(w));
}
template <> QS_DEVINL float2 pair_to_float2<Dt::F16>(uint32_t w) {
    return make_float2(f16lo(w), f16hi(w));
}

// Scalar element load of a float dtype (slow path helpers; q loads only).
template <Dt T> QS_DEVINL float load_elem(const void* p, size_t i);
template <> QS_DEVINL float load_elem<Dt::F32>(const void* p, size_t i) {
    return static_cast<const float*>(p)[i];
}
template <> QS_DEVINL float load_elem<Dt::BF16>(const void* p, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
}
template <> QS_DEVINL float load_elem<Dt::F16>(const void* p, size_t i) {
    return __half2float(__ushort_as_half(static_cast<const unsigned short*>(p)[i]));
}

// q loader with a runtime dtype (q is tiny; the branch is uniform).
QS_DEVINL float load_q(const void* q, int dt, size_t i) {
    if (dt == QS_BF16) return load_elem<Dt::BF16>(q, i);
    if (dt == QS_F16) return load_elem<Dt::F16>(q, i);
    return load_elem<Dt::F32>(q, i);
}

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------

// 16-byte streaming load that bypasses L1 allocation (each byte used once).
QS_DEVINL uint4 ldg_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

QS_DEVINL void stg_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Loads issued exactly where they stand (asm volatile: the compiler may not
// sink them below a branch on an earlier load), so that round trips that do
// not depend on one another overlap.  Read-only data only.
QS_DEVINL int32_t ldg_now_s32(const int32_t* p) {
    int32_t v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
QS_DEVINL uint32_t ldg_now_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
QS_DEVINL uint32_t ldg_now_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
QS_DEVINL uint2 ldg_now_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
QS_DEVINL uint4 ldg_now_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
// Raw bits of q element i (fp32: the word; 16-bit: the half-word) and their
// value; split so that the load is issued before a branch and converted after.
QS_DEVINL uint32_t ldg_now_q_bits(const void* q, int dt, size_t i) {
    return dt == QS_F32 ? ldg_now_u32(static_cast<const float*>(q) + i)
                        : ldg_now_u16(static_cast<const uint16_t*>(q) + i);
}
QS_DEVINL float q_bits_value(uint32_t w, int dt) {
    if (dt == QS_F32) return __uint_as_float(w);
    if (dt == QS_BF16) return __uint_as_float(w << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w)));
}

// L2-coherent loads for data written by other CTAs of the same grid.
QS_DEVINL float ldcg_f32(const float* p) { return __ldcg(p); }

// ---------------------------------------------------------------------------
// packed fp32x2 arithmetic (sm_100 family)
// ---------------------------------------------------------------------------

QS_DEVINL unsigned long long pack2(float lo, float hi) {
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
QS_DEVINL float2 unpack2(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}
// d = a * b + c, elementwise on two fp32 lanes, each rounded once.
QS_DEVINL unsigned long long fma2(unsigned long long a, unsigned long long b,
                                  unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
QS_DEVINL unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 2^x on the SFU (hardware approximation, ~2 ulp); -inf -> 0.
QS_DEVINL float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// ordering keys
// ---------------------------------------------------------------------------

// Monotone map of a float onto uint32 (larger float -> larger key).  -0 is
// folded onto +0 first so that equal scores get equal keys.
QS_DEVINL uint32_t float_key(float f) {
    f = f + 0.0f;
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// shared-memory addresses and launch controls (inline PTX)
// ---------------------------------------------------------------------------

QS_DEVINL uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch controls.
QS_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QS_DEVINL void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace qs

// ---------------------------------------------------------------------------
// host helpers (defined in qs_api.cu)
// ---------------------------------------------------------------------------
namespace qs {
int num_sms();                      // of the current device (cached per device)
cudaError_t last_launch_error();
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the attribute is set once per (kernel, device) so that
// later calls -- including ones made under stream capture -- do no driver work.
bool ensure_smem(const void* func, size_t bytes);
}  // namespace qs

#define QS_CHECK_LAUNCH()                                   \
    do {                                                    \
        if (qs::last_launch_error() != cudaSuccess) return QS_ECUDA; \
    } while (0)
