// Device helpers shared by the kernels of liblsa: bulk-copy staging with
// mbarriers (inline PTX for sm_103a), bf16 / e4m3 conversions, bounded waits
// and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "lsa_internal.h"

namespace lsa {

// ---------------------------------------------------------------- status

// Kernels record data errors by setting bit `code` of the per-device status
// word (never by faulting): the offending access is skipped.
__device__ __forceinline__ void flag_error(uint32_t *status, int code)
{
    if (status) atomicOr(status, 1u << code);
}

// ---------------------------------------------------------------- counters between CTAs

// red.release / ld.acquire of a GPU-scope counter.
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until *p == want (acquire).  Gives up after `budget` SM clock
// cycles, records LSA_ERR_TIMEOUT and returns false: a wait never hangs.
// The counters it waits on only ever reach `want` once per call and stay
// there until every waiter has passed, so an exact comparison cannot miss.
__device__ __forceinline__ bool wait_counter_eq(const uint32_t *p, uint32_t want, uint32_t *status, long long budget)
{
    if (ld_acquire(p) == want) return true;
    const long long t0 = clock64();
    while (ld_acquire(p) != want) {
        if (clock64() - t0 > budget) {
            flag_error(status, LSA_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(100);
    }
    return true;
}

// Every thread of the CTA calls this once its results are written; it
// returns true in every thread of the group's last CTA to arrive (`members`
// CTAs share the counter), which may then read what the others wrote.  The
// caller resets the counter.
__device__ __forceinline__ bool last_cta_arrival(uint32_t *counter, uint32_t members, uint32_t *s_flag)
{
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(counter, 1u);
        *s_flag = prev == members - 1 ? 1u : 0u;
    }
    __syncthreads();
    const bool last = *s_flag != 0u;
    if (last) __threadfence();
    return last;
}

// ---------------------------------------------------------------- dependent launch

// A kernel launched with programmatic stream serialization (a dependent)
// may start once every CTA of the kernel before it has signalled
// launch_dependents; it must wait (griddepcontrol.wait: that kernel has
// completed and its writes are visible) before it reads that kernel's
// results.  Outside a dependent launch the wait returns at once.  Kernels
// call pdl_enter at their top: the wait first, so that as dependents they
// run nothing before their predecessor completes, then the signal, so that
// their own dependents start only once everything before them on the
// stream has completed.  The decode step's attention kernel signals first
// and waits after its set-up (attention_flat.cu).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait();
    pdl_launch_dependents();
}

// pdl_mode / pdl_enabled: lsa_internal.h

// dependent: launch with programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_ex(bool dependent, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_step_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               Args &&...args)
{
    return launch_kernel_ex(pdl_enabled(), kern, grid, block, smem, s, static_cast<Args &&>(args)...);
}

// A launch in thread-block clusters of cs CTAs along x (grid.x a multiple
// of cs); sizes above 8 need the kernel's non-portable-size attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_kernel(bool dependent, int cs, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = dependent ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// How many clusters of cs CTAs of the kernel can be resident at once (0:
// none, or the query failed).  Sets the non-portable-size attribute first
// when cs > 8, and the dynamic shared memory limit to smem.
template <typename... KArgs>
int max_active_clusters(void (*kern)(KArgs...), int cs, dim3 block, size_t smem)
{
    if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// ---------------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Barrier over every thread of every CTA of the cluster; the CTA's shared
// memory writes before it are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the shared::cta address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Two 32-bit words to an 8-byte aligned shared::cluster address in one store.
__device__ __forceinline__ void st_cluster_v2_u32(uint32_t a, uint32_t x, uint32_t y)
{
    asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void red_cluster_add_u32(uint32_t a, uint32_t v)
{
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ double ld_cluster_f64(uint32_t a)
{
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(a) : "memory");
    return v;
}

// ---------------------------------------------------------------- smem / mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  Gives up after `budget` clock cycles
// (records LSA_ERR_TIMEOUT) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                          long long budget)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) {
            flag_error(status, LSA_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Tiled 2-D tensor copy (TMA) global -> shared: the tensor map's box at
// element coordinates (x, y) into dst (shared address), with the map's
// swizzle; completion is counted in bytes on the mbarrier at bar.  tmap:
// the generic address of a __grid_constant__ CUtensorMap parameter.  x times
// the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy (TMA engine) global -> shared; completion is counted in
// bytes on `bar`.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---------------------------------------------------------------- conversions

// Two packed bf16 (low half = element 0) -> two floats.  bf16 is the upper
// half of a binary32, so this is exact.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u)
{
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ float bf_to_f(uint16_t u)
{
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// fp64 -> bf16 with a single round-to-nearest-even: first round toward zero
// to binary32 and make the result "sticky" (round to odd: set the last bit if
// anything was discarded), then round binary32 -> bf16 to nearest even.
// Rounding to odd with at least two extra bits and then to nearest gives the
// correctly rounded result (Boldo & Melquiond, "Emulation of FMA and
// correctly rounded sums: proved algorithms using rounding to odd", 2008).
__device__ __forceinline__ uint16_t f64_to_bf16_rne(double x)
{
    float f = __double2float_rz(x);
    if (static_cast<double>(f) != x && !isnan(x) && !isinf(f)) {
        f = __uint_as_float(__float_as_uint(f) | 1u);
    }
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Two e4m3 bytes (low byte = element 0) -> two floats; every e4m3 value is
// exact in half precision.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t two)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    __half2 hh = *reinterpret_cast<__half2 *>(&h2);
    return __half22float2(hh);
}

// Order-preserving map from fp32 to uint32 for the radix select: larger
// float -> larger key.  -0 is first made +0.  Keys of finite values and of
// +inf are > 0x007fffff; the caller reserves 0 for "not a candidate".
__device__ __forceinline__ uint32_t float_to_key(float s)
{
    uint32_t b = __float_as_uint(s);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of float_to_key on the keys it produces.
__device__ __forceinline__ float key_to_float(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ---------------------------------------------------------------- loads

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------- L2 policy for bulk streams

// The summaries and the K/V a step streams are read once: loads of them
// carry an L2 evict-first policy so that they do not push out what is read
// again soon (page tables, lengths, the score rows, the kernels' code).
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ldg_stream_v4(const void *p, uint64_t pol)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// ---------------------------------------------------------------- async copies

// 16-byte cp.async (LSU path) into shared memory; completion by commit
// groups.  Unlike the bulk-copy engine, which serves one issuing warp's
// copies one after another, these overlap freely across lanes and warps.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// cp_async16 with an L2 cache policy (l2_evict_first for bulk streams).
// 4-byte cp.async (L1-allocating form): dst and src 4-byte aligned.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async16_policy(uint32_t dst, const void *src, uint64_t pol)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}

// Pulls the 128-byte line holding p into L1 (no register result).
__device__ __forceinline__ void prefetch_l1(const void *p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- tensor-core fragments

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A * B for one m16n8k16 tile (bf16 in, fp32 accumulate); rows 8..15 of
// A are zero (a1 = a3 = 0): the GQA group occupies rows 0..7 at most.
__device__ __forceinline__ void mma_bf16_rows8(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Hardware base-2 exponential / logarithm (approximate, ~2 ulp).
__device__ __forceinline__ float fast_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fast_lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk `ch` of token row `t` (0..15) inside a tile
// of 16 rows stored as 128-byte-wide sub-tiles with the XOR swizzle
// (chunk ^ row%8): 8 rows read at one column hit 8 different bank groups.
__device__ __forceinline__ uint32_t swizzle_offset(int t, int ch)
{
    return (uint32_t)((ch >> 3) * (16 * 128) + t * 128 + (((ch & 7) ^ (t & 7)) << 4));
}

// ---------------------------------------------------------------- tcgen05 (fifth-generation tensor cores)

// Tensor memory (TMEM) is 128 lanes x 512 columns of 32-bit cells per SM.
// An address is (lane << 16) | column.  Allocation is by a whole warp, in
// power-of-two column counts >= 32; the base address is written to shared
// memory.  Every allocation must be freed by the same CTA before it exits.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations across a thread barrier.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Makes this thread's generic-proxy writes to shared memory (st.shared,
// cp.async) visible to the async proxy that tcgen05.mma reads through.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Byte offset of 16-byte chunk j (0..7) of row t inside an atom column of
// 8-row x 128-byte atoms with the 128-byte swizzle.
__device__ __forceinline__ uint32_t atom_offset(int t, int j)
{
    return (uint32_t)((t >> 3) * 1024 + (t & 7) * 128 + ((j ^ (t & 7)) << 4));
}

// Shared-memory matrix descriptor with the 128-byte swizzle: atoms of 8
// rows x 128 bytes (1024-byte aligned), the 16-byte chunk index of each row
// XORed with the row index (swizzle_offset above lays tiles out this way).
// lbo / sbo: byte offsets between atoms along the leading and the strided
// dimension; bits 46-47 hold the descriptor version (1), bits 61-63 the
// layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulation:
// D format bits 4-5, A and B formats bits 7-9 / 10-12, A and B major-ness
// bits 15 / 16 (0 = K-major, 1 = MN-major), N / 8 in bits 17-22, M / 16 in
// bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; issued by one thread.  A's M rows are
// TMEM lanes and its K elements run along the columns, two 16-bit elements
// a 32-bit column (a K = 16 step spans 8 columns from a_tmem).
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// One arrive on `bar` once every tcgen05.mma this thread issued before it
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Writes 32 consecutive columns of this thread's TMEM lane from registers
// (the warp writes the 32 lanes of its quadrant: taddr's lane field is 32 *
// (warp % 4)).  tmem_st_wait makes them complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive columns of this thread's TMEM lane (the warp reads the 32
// lanes of its quadrant: taddr's lane field is 32 * (warp % 4)).  The wait
// for the load is part of the same statement, so no use of the registers
// can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace lsa
