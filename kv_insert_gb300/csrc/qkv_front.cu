// libqkvfront: the decode-batch QKV front as one sm_103a kernel.
//
// What it computes is stated in include/qkvfront.h.  Sources: the API pages
// "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.attention.qkv_front"
// (module docstring: projection, weightless RMS norm, interleaved RoPE, y
// store, paged K/V insert in one launch; summaries of QkvFrontKernel.produce,
// consume, aux, send, finish) and "...runtime.cute_ops" (split_qkv row
// layout, supports_call, unsupported_projection; attn2 paragraph for the
// cache layout).
//
// Kernel design (one CTA per head and K split, a cluster per head when K is
// split):
//   - grid (splits, N / 64); CTA (r, h) owns head h (W rows 64h..64h+63) and
//     the K stages r, r + splits, r + 2 splits, ... (cyclic stripes);
//   - warp 4 lane 0 (producer) streams 64 x 64 bf16 W boxes and the matching
//     token x 64 x boxes into a `stages`-deep shared-memory ring with TMA
//     (128-byte swizzle), issuing the first ring's worth of W before the PDL
//     wait (W is never written by a kernel in flight);
//   - warps 0..3 (consumers) run mma.sync m16n8k16 bf16 -> fp32 with the W
//     rows as the M side (16 rows per warp) and the tokens as the N side
//     (one or two 8-token tiles), reading fragments with ldmatrix;
//   - warp 5 (aux) loads the tokens' positions, slots and cos|sin rows after
//     the PDL wait and checks them against the table and cache sizes;
//   - the FP32 partials go to shared memory; with splits > 1 the owner CTA of
//     token t (cluster rank t % splits) reads all ranks' partials through
//     distributed shared memory and sums them in rank order 0, 1, ..., so the
//     result depends only on the launch shape (no atomics, no global
//     scratch);
//   - the epilogue rounds to BF16, norms and rotates q and k heads (one lane
//     per RoPE pair), stores the row and writes K / V into the paged cache.
//
// Every shared-memory barrier wait is bounded in time: on expiry the CTA
// raises QKVF_STATUS_WAIT_TIMEOUT in a device status word, stops waiting,
// drains its own copies in flight and exits normally.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "qkvfront.h"

namespace qkvf {

constexpr int kHidden = 8192;        // hidden size (page qkv_front, hidden_rows_ok: [rows, 8192])
constexpr int kHeadDim = 64;         // one head = 64 output columns (module docstring)
constexpr int kQPerKv = 8;           // q (and gate) heads per KV head (cute_ops, split_qkv)
constexpr int kPageSlots = 16;       // cache [pages, num_kv_heads, 16, 128] (cute_ops, attn2)
constexpr int kSlotWidth = 128;      // K | V per slot
constexpr int kMaxTokens = 16;       // 1 <= M <= 16 (module docstring)
constexpr int kBoxK = 64;            // k per TMA box row: 128 bytes = one swizzle row
constexpr int kBoxBytesW = 64 * 128; // W box: 64 rows x 128 bytes
constexpr int kConsumerWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kAuxWarp = 5;
constexpr int kWarps = 6;
constexpr int kThreads = kWarps * 32;
constexpr int kPartStride = 68;      // floats per token row of the partial (64 + 4: no bank conflicts)
constexpr float kEps = 1e-6f;
constexpr int kMaxSmemPerCta = 232448;   // 227 KB opt-in limit
constexpr int kSmemPerSm = 233472;       // 228 KB per SM
constexpr int kSmemReservedPerCta = 1024;

enum HeadKind { kQ = 0, kK = 1, kV = 2, kGate = 3 };

__device__ unsigned int g_status;

struct FrontParams {
    const uint16_t *W;   // [N, 8192] (the resident engine loads part of its share with plain loads)
    const int64_t *positions;
    const int64_t *slots;
    const float *cos_sin;
    uint16_t *out;
    uint16_t *kv_cache;
    int64_t cos_rows;
    int64_t num_pages;
    unsigned long long wait_limit_ns;
    int M;
    int N;
    int nkv;
    int splits;
    int stages;
    int kb;           // 64-k boxes per ring stage (1, 2 or 4)
    int l2_prefetch;  // ring stages of W prefetched into L2 before the PDL wait
};

// Shared-memory layout of one CTA, from the base (1024-byte aligned).  The
// FP32 partials reuse the start of the W ring: they are written only after
// every consumer warp has finished reading the ring.
struct Layout {
    uint32_t w, x, full, empty, done, tmem_slot, part, pos, slot, cs, flag, abort_flag, total;
};

__host__ __device__ inline Layout layout_of(int mt, int kb, int stages)
{
    Layout L;
    uint32_t off = 0;
    L.w = off;
    L.part = off;
    off += (uint32_t)stages * kb * kBoxBytesW;
    L.x = off;
    off += (uint32_t)stages * kb * mt * 128;
    L.full = off;
    off += (uint32_t)stages * 8;
    L.empty = off;
    off += (uint32_t)stages * 8;
    L.done = off;
    off += 8;
    L.tmem_slot = off;
    off += 8;
    off = (off + 15u) & ~15u;
    // per-token arrays for the tile's mt tokens (M <= mt)
    L.pos = off;
    off += (uint32_t)mt * 8;
    L.slot = off;
    off += (uint32_t)mt * 8;
    L.cs = off;
    off += (uint32_t)mt * kHeadDim * 4;
    L.flag = off;
    off += (uint32_t)mt * 4;
    L.abort_flag = off;
    off += 16;
    L.total = off;
    return L;
}

// dynamic shared memory to request: the layout plus slack to align the base
__host__ __device__ inline uint32_t smem_bytes(int mt, int kb, int stages)
{
    return layout_of(mt, kb, stages).total + 1024;
}

// ---- PTX helpers -----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the barrier's phase with this parity completes, for at most
// limit_ns.  On expiry: raise the status bit, set the CTA's abort flag and
// return false.  With `honour_abort`, also return false as soon as another
// thread of the CTA has aborted.
__device__ __noinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long limit_ns, bool honour_abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long start = global_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (honour_abort && *abort_flag) return false;
        if (global_ns() - start > limit_ns) {
            *abort_flag = 1;
            atomicOr(&g_status, QKVF_STATUS_WAIT_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled TMA load (k within a 64-k block, rows, 64-k blocks): one copy
// brings a ring stage's kb boxes.  c0 is always 0.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0, int c1,
                                            int c2, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

// Prefetch one stage of W into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *m, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void consumer_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// ---- tcgen05 (5th-generation tensor core, accumulator in tensor memory) ----

// Shared-memory matrix descriptor of a K-major operand stored as TMA wrote it
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address / 16
    d |= (uint64_t)1 << 16;                             // leading offset (unused when swizzled)
    d |= (uint64_t)(1024u >> 4) << 32;                  // stride offset: one 8-row group
    d |= (uint64_t)1 << 46;                             // descriptor version
    d |= (uint64_t)2 << 61;                             // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: BF16 A and B, FP32 accumulator, both
// operands K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

constexpr uint32_t kTmemCols = 32;   // smallest allocation; the accumulator needs 8 or 16 columns

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kTmemCols)
                 : "memory");
}

// 32 lanes x 8 (or 16) consecutive 32-bit columns of tensor memory: thread i
// of the warp gets lane (taddr.lane + i), columns taddr.col .. +7 (+15).
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n"
        "barrier.cluster.wait.acquire.aligned;\n" ::
            : "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 lo, __nv_bfloat16 hi)
{
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// ---- the q / k head epilogue (shared by both kernels) ----------------------
// Lane l holds the BF16 values (f0, f1) of head columns 2l, 2l+1 and the
// cos / sin of pair l.  Weightless RMS norm over the 64 columns (butterfly sum:
// every lane ends with the same bits), then the interleaved rotation of the
// lane's pair, rounded to BF16.  The whole warp must call it.
__device__ __forceinline__ uint32_t qk_norm_rope_pair(float f0, float f1, float c, float sn)
{
    float ss = __fadd_rn(__fmul_rn(f0, f0), __fmul_rn(f1, f1));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    const float ms = __fdiv_rn(ss, (float)kHeadDim);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, kEps)));
    const float a = __fmul_rn(f0, r), b = __fmul_rn(f1, r);
    const float y0 = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, sn));
    const float y1 = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, sn));
    return pack_bf16x2(__float2bfloat16_rn(y0), __float2bfloat16_rn(y1));
}

// The finish of token u's 64 columns of head `head`: lane l holds the FP32
// sums (v.x, v.y) of columns 2l, 2l+1.  Round to BF16; for q and k heads the
// norm and RoPE with the position's (c, sn) of pair l; store the row segment;
// for k and v heads write the slot's K or V half.  flag bit 0: the position
// is in the table (else a q / k head writes nothing); bit 1: the token
// inserts.  The whole warp calls it (the norm shuffles across lanes).
__device__ __forceinline__ void finish_pair(const FrontParams &p, int head, int kind, int u, int lane,
                                            float2 v, int flag, float c, float sn, int64_t slot)
{
    const __nv_bfloat16 p0 = __float2bfloat16_rn(v.x);
    const __nv_bfloat16 p1 = __float2bfloat16_rn(v.y);
    uint32_t word;
    if (kind == kQ || kind == kK) {
        if (!(flag & 1)) return;   // no table row for this position: nothing written
        word = qk_norm_rope_pair(__bfloat162float(p0), __bfloat162float(p1), c, sn);
    } else {
        word = pack_bf16x2(p0, p1);
    }
    uint32_t *orow = reinterpret_cast<uint32_t *>(p.out + (size_t)u * p.N + (size_t)head * kHeadDim);
    orow[lane] = word;
    if ((kind == kK || kind == kV) && (flag & 2)) {
        const int64_t page = slot / kPageSlots, offs = slot % kPageSlots;
        const int gkv = head - kQPerKv * p.nkv - (kind == kV ? p.nkv : 0);
        uint16_t *dst = p.kv_cache + ((page * p.nkv + gkv) * kPageSlots + offs) * kSlotWidth +
                        (kind == kV ? kHeadDim : 0);
        reinterpret_cast<uint32_t *>(dst)[lane] = word;
    }
}

// ---- the front kernel ------------------------------------------------------

// TC: the contraction runs on tcgen05 (one thread issues M=64 x N=MT x K=16
// MMAs from the ring into a tensor-memory accumulator); otherwise on
// mma.sync in the four consumer warps.
template <int MT, bool TC>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_front_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const FrontParams p)
{
    constexpr int NT = MT / 8;                       // 8-token mma column tiles
    constexpr uint32_t kBoxBytesX = MT * 128;
    const int KB = p.kb;
    const uint32_t kStageTx = (uint32_t)KB * (kBoxBytesW + kBoxBytesX);
    const int kStepsAll = kHidden / (kBoxK * KB);

    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    const Layout L = layout_of(MT, KB, p.stages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.splits;
    const uint32_t rank = S > 1 ? cluster_rank() : 0u;
    const int head = blockIdx.y;
    const int steps = kStepsAll / S;
    const int stages = p.stages;

    const uint32_t sW = smem_u32(smem + L.w);
    const uint32_t sX = smem_u32(smem + L.x);
    const uint32_t full0 = smem_u32(smem + L.full);
    const uint32_t empty0 = smem_u32(smem + L.empty);
    const uint32_t done_bar = smem_u32(smem + L.done);
    float *part = reinterpret_cast<float *>(smem + L.part);
    int64_t *s_pos = reinterpret_cast<int64_t *>(smem + L.pos);
    int64_t *s_slot = reinterpret_cast<int64_t *>(smem + L.slot);
    float *s_cs = reinterpret_cast<float *>(smem + L.cs);
    int *s_flag = reinterpret_cast<int *>(smem + L.flag);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.abort_flag);

    const int q_heads = kQPerKv * p.nkv;
    const int kind = head < q_heads ? kQ : head < q_heads + p.nkv ? kK
                   : head < q_heads + 2 * p.nkv ? kV : kGate;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            // released by the MMA issuer's commit (TC) or by each consumer warp
            mbar_init(empty0 + 8 * s, TC ? 1 : kConsumerWarps);
        }
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_barrier_init();
        // Dependents may launch now: before their own PDL wait they read only
        // their weights, which this kernel never writes.
        griddep_launch_dependents();
    }
    if constexpr (TC) {
        __syncwarp();
        if (warp == 0) tmem_alloc(smem_u32(smem + L.tmem_slot));   // whole warp, converged
        tc_fence_before();
    }
    __syncthreads();
    if constexpr (TC) tc_fence_after();
    const uint32_t tmem_d = TC ? *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot) : 0u;

    if (warp == kProducerWarp) {
        // ---- produce: the W / x ring ------------------------------------
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();   // streamed once
            const uint64_t pol_x = policy_evict_last();    // re-read by every CTA
            tma_prefetch_map(&tmW);
            tma_prefetch_map(&tmX);
            const int row0 = head * kHeadDim;
            const int npre = steps < stages ? steps : stages;
            // one copy per stage for W and one for x: the maps are 3-D
            // (k, rows, 64-k blocks) with a box of the stage's kb blocks
            for (int i = 0; i < npre; ++i) {
                const int j = (int)rank + i * S;
                mbar_expect_tx(full0 + 8 * i, kStageTx);
                tma_load_3d(sW + (uint32_t)(i * KB) * kBoxBytesW, &tmW, full0 + 8 * i, 0, row0, j * KB, pol_w);
            }
            // weights further ahead into L2 while the previous kernel finishes
            const int pf_end = npre + p.l2_prefetch < steps ? npre + p.l2_prefetch : steps;
            for (int i = npre; i < pf_end; ++i) tma_prefetch_l2_3d(&tmW, 0, row0, ((int)rank + i * S) * KB);
            griddep_wait();   // x is written by the kernel before this one
            for (int i = 0; i < npre; ++i) {
                const int j = (int)rank + i * S;
                tma_load_3d(sX + (uint32_t)(i * KB) * kBoxBytesX, &tmX, full0 + 8 * i, 0, 0, j * KB, pol_x);
            }
            int issued = npre;
            int s = npre == stages ? 0 : npre;
            int use = npre == stages ? 1 : 0;   // how many times slot s was filled before
            for (int i = npre; i < steps; ++i) {
                if (!bounded_wait(empty0 + 8 * s, (uint32_t)((use - 1) & 1), s_abort,
                                  p.wait_limit_ns, true))
                    break;
                const int j = (int)rank + i * S;
                mbar_expect_tx(full0 + 8 * s, kStageTx);
                tma_load_3d(sW + (uint32_t)(s * KB) * kBoxBytesW, &tmW, full0 + 8 * s, 0, row0, j * KB, pol_w);
                tma_load_3d(sX + (uint32_t)(s * KB) * kBoxBytesX, &tmX, full0 + 8 * s, 0, 0, j * KB, pol_x);
                ++issued;
                if (++s == stages) {
                    s = 0;
                    ++use;
                }
            }
            if (*s_abort) {
                // drain: every copy this CTA issued lands before it exits
                const int first = issued > stages ? issued - stages : 0;
                for (int i = first; i < issued; ++i)
                    bounded_wait(full0 + 8 * (i % stages), (uint32_t)((i / stages) & 1), s_abort,
                                 p.wait_limit_ns, false);
            }
        }
        __syncwarp();
        griddep_wait();
    } else if (warp == kAuxWarp) {
        // ---- aux: the epilogue's per-token inputs -------------------------
        griddep_wait();
        unsigned bad = 0u;
        if (lane < p.M) {
            const int64_t pos = p.positions[lane];
            const int64_t slot = p.slots[lane];
            const int64_t slot_end = p.num_pages * (int64_t)kPageSlots;
            const bool pos_ok = pos >= 0 && pos < p.cos_rows;
            const bool slot_over = slot >= slot_end;
            const bool insert = slot >= 0 && !slot_over && pos_ok;
            s_pos[lane] = pos;
            s_slot[lane] = slot;
            s_flag[lane] = (pos_ok ? 1 : 0) | (insert ? 2 : 0);
            bad = (pos_ok ? 0u : QKVF_STATUS_BAD_POSITION) | (slot_over ? QKVF_STATUS_BAD_SLOT : 0u);
        }
        // one report per call: the warp's OR, from one CTA
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0 && bad != 0u && head == 0 && rank == 0) atomicOr(&g_status, bad);
        __syncwarp();
        if (kind == kQ || kind == kK) {
            for (int t = (int)rank; t < p.M; t += S) {
                if (!(s_flag[t] & 1)) continue;
                const float2 v =
                    reinterpret_cast<const float2 *>(p.cos_sin + s_pos[t] * kHeadDim)[lane];
                reinterpret_cast<float2 *>(s_cs + t * kHeadDim)[lane] = v;
            }
        }
    } else if constexpr (TC) {
        // ---- consume (tcgen05): one thread issues every MMA -----------------
        griddep_wait();
        if (warp == 0 && lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(64, MT);
            int s = 0;
            uint32_t phase = 0;
            for (int i = 0; i < steps; ++i) {
                if (mbar_try_wait(full0 + 8 * s, phase) ||
                    bounded_wait(full0 + 8 * s, phase, s_abort, p.wait_limit_ns, true)) {
                    tc_fence_after();
                    for (int b = 0; b < KB; ++b) {
                        const uint32_t wbox = sW + (uint32_t)(s * KB + b) * kBoxBytesW;
                        const uint32_t xbox = sX + (uint32_t)(s * KB + b) * kBoxBytesX;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)   // K = 16 per MMA: 32 bytes along the row
                            umma_bf16(tmem_d, umma_desc_sw128(wbox + 32u * kk),
                                      umma_desc_sw128(xbox + 32u * kk), idesc,
                                      (i | b | kk) != 0 ? 1u : 0u);
                    }
                }
                umma_commit(empty0 + 8 * s);   // the slot is free once these MMAs have read it
                if (++s == stages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            umma_commit(done_bar);
        }
        __syncwarp();
        // The M = 64 accumulator holds rows 16w..16w+15 in lanes 0..15 of
        // tensor-memory sub-partition w; warp w reads its own sub-partition.
        const bool ready = mbar_try_wait(done_bar, 0) ||
                           bounded_wait(done_bar, 0, s_abort, p.wait_limit_ns, false);
        __syncwarp();
        tc_fence_after();
        const uint32_t taddr = tmem_d + ((uint32_t)(warp * 32) << 16);
        uint32_t r[MT];
#pragma unroll
        for (int i = 0; i < MT; ++i) r[i] = 0u;
        // a timed-out wait leaves the MMAs possibly running: the accumulator
        // is not read (the call's outputs are invalid and flagged anyway)
        if (__all_sync(0xffffffffu, ready)) {
            if constexpr (MT == 8)
                tmem_ld_x8(taddr, r);
            else
                tmem_ld_x16(taddr, r);
            tmem_ld_wait();
        }
        if (lane < 16) {
#pragma unroll
            for (int tok = 0; tok < MT; ++tok)
                part[tok * kPartStride + warp * 16 + lane] = __uint_as_float(r[tok]);
        }
    } else {
        // ---- consume: mma.sync over the ring ------------------------------
        griddep_wait();
        // one accumulator set per k16 step of a box: four independent mma
        // chains instead of one serial chain (mma.sync latency, not issue
        // rate, is what limits a single chain); summed in a fixed order at the end
        float acc[NT][4][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[nt][kk][r] = 0.f;

        // ldmatrix row addresses.  A: lane l feeds row (l & 7) + 8 ((l >> 3) & 1)
        // of this warp's 16 W rows, 16-byte chunk (l >> 4) of the k16 step.
        // B: lane l feeds token (l & 7) (+ 8 (l >> 4) with two tiles), chunk
        // ((l >> 3) & 1).  The 128-byte swizzle XORs the chunk with row % 8.
        const uint32_t a_row = (uint32_t)(warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8);
        const uint32_t a_off = a_row * 128u;
        const uint32_t a_hi = (uint32_t)(lane >> 4);
        const uint32_t b_tok = NT == 2 ? (uint32_t)((lane & 7) + ((lane >> 4) << 3))
                                       : (uint32_t)(lane & 7);
        const uint32_t b_off = b_tok * 128u;
        const uint32_t b_hi = (uint32_t)((lane >> 3) & 1);
        const uint32_t sw = (uint32_t)(lane & 7);   // row % 8 for both operands

        int s = 0;
        uint32_t phase = 0;
        for (int i = 0; i < steps; ++i) {
            // every lane waits (each gets the barrier's acquire); the warp
            // then agrees, so ldmatrix / mma always run on a converged warp
            const bool landed = mbar_try_wait(full0 + 8 * s, phase) ||
                                bounded_wait(full0 + 8 * s, phase, s_abort, p.wait_limit_ns, true);
            if (__all_sync(0xffffffffu, landed)) {
                for (int b = 0; b < KB; ++b) {
                    const uint32_t wbox = sW + (uint32_t)(s * KB + b) * kBoxBytesW;
                    const uint32_t xbox = sX + (uint32_t)(s * KB + b) * kBoxBytesX;
                    uint32_t a[4][4], bb[4][4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        ldsm_x4(wbox + a_off + ((((uint32_t)(2 * kk) + a_hi) ^ sw) << 4), a[kk][0],
                                a[kk][1], a[kk][2], a[kk][3]);
                        const uint32_t baddr =
                            xbox + b_off + ((((uint32_t)(2 * kk) + b_hi) ^ sw) << 4);
                        if constexpr (NT == 2)
                            ldsm_x4(baddr, bb[kk][0], bb[kk][1], bb[kk][2], bb[kk][3]);
                        else
                            ldsm_x2(baddr, bb[kk][0], bb[kk][1]);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        mma_bf16_16816(acc[0][kk], a[kk][0], a[kk][1], a[kk][2], a[kk][3],
                                       bb[kk][0], bb[kk][1]);
                        if constexpr (NT == 2)
                            mma_bf16_16816(acc[1][kk], a[kk][0], a[kk][1], a[kk][2], a[kk][3],
                                           bb[kk][2], bb[kk][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
            if (++s == stages) {
                s = 0;
                phase ^= 1u;
            }
        }
        float sum[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                sum[nt][r] = __fadd_rn(__fadd_rn(acc[nt][0][r], acc[nt][1][r]),
                                       __fadd_rn(acc[nt][2][r], acc[nt][3][r]));
        // the partials overwrite the ring: every consumer warp must be done with it
        consumer_bar_sync();
        // accumulator fragment: c0 (row g, token 2t), c1 (g, 2t+1),
        // c2 (g+8, 2t), c3 (g+8, 2t+1) with g = lane / 4, t = lane % 4
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int tok = nt * 8 + 2 * t;
            const int col = warp * 16 + g;
            part[tok * kPartStride + col] = sum[nt][0];
            part[(tok + 1) * kPartStride + col] = sum[nt][1];
            part[tok * kPartStride + col + 8] = sum[nt][2];
            part[(tok + 1) * kPartStride + col + 8] = sum[nt][3];
        }
    }
    if constexpr (TC) tc_fence_before();
    __syncthreads();
    if constexpr (TC) {
        if (warp == 0) {   // every tensor-memory read is done
            // and every issued MMA: the issuer (lane 0 of this warp) committed
            // done_bar before this point, so after a timed-out wait above the
            // MMAs still end within the bounded wait here
            if (!mbar_try_wait(done_bar, 0)) bounded_wait(done_bar, 0, s_abort, p.wait_limit_ns, false);
            __syncwarp();
            tc_fence_after();
            tmem_dealloc(tmem_d);
        }
    }
    if (S > 1) cluster_sync_all();   // every rank's partial is in its shared memory

    // ---- finish: reduce, round, norm, RoPE, store, insert -------------------
    const uint32_t part_addr = smem_u32(part);
    for (int li = warp;; li += kWarps) {
        const int u = (int)rank + li * S;   // tokens owned by this rank: u % S == rank
        if (u >= p.M) break;
        float2 v;
        if (S == 1) {
            v = reinterpret_cast<const float2 *>(part + u * kPartStride)[lane];
        } else {
            // every rank's partial is requested before the first add (one
            // round trip, not S); the adds keep rank order 0..S-1
            const uint32_t a = part_addr + (uint32_t)(u * kPartStride + 2 * lane) * 4u;
            float2 r[16];
#pragma unroll
            for (int src = 0; src < 16; ++src)
                if (src < S) r[src] = ld_cluster_f2(map_to_rank(a, (uint32_t)src));
            v = r[0];
#pragma unroll
            for (int src = 1; src < 16; ++src) {
                if (src < S) {
                    v.x = __fadd_rn(v.x, r[src].x);
                    v.y = __fadd_rn(v.y, r[src].y);
                }
            }
        }
        // norm and RoPE of pair (2 lane, 2 lane + 1): cos in column lane, sin
        // in column 32 + lane of the position's row
        const bool qk = kind == kQ || kind == kK;
        finish_pair(p, head, kind, u, lane, v, s_flag[u], qk ? s_cs[u * kHeadDim + lane] : 0.f,
                    qk ? s_cs[u * kHeadDim + 32 + lane] : 0.f, s_slot[u]);
    }
    if (S > 1) cluster_sync_all();   // no CTA leaves while its partial may still be read
}

// ---- the resident front: a CTA's whole weight share on chip before the wait --
//
// For a small projection (N = 1152: 18 heads, K split 8 ways, 128 KB of W per
// CTA) the call is short enough that the time after the PDL wait decides it.
// Here every byte of W a CTA needs is on chip before that wait, in the
// previous call's shadow: stages 0 and 1 (64 KB) in shared memory through one
// 4-D TMA copy, stages 2 and 3 (64 KB) in the registers of the four warps
// through 16-byte loads.  After the wait one TMA copy brings the CTA's x
// stripe; the warps contract it with both halves (mma.sync), and each CTA
// pushes its FP32 partial of token u to the owner rank u % S with st.async,
// completing on the owner's barrier.  The owner adds the S partials in rank
// order 0..S-1 (the same fixed order for every launch) and runs the finish;
// the other CTAs exit as soon as their partials are sent.
//
// Register stages use a k order of their own inside each 32-k chunk: lane
// (g, t) holds W[row][c + 8t .. c + 8t + 7] (one 16-byte load) and feeds it
// to two k16 steps, the first taking k c + 8t + {0,1,2,3}, the second
// c + 8t + {4,5,6,7}; the x fragment takes the same k from shared memory.
// A dot product may visit its k in any order, so only the FP32 summation
// order differs from a ring stage.

constexpr int kResThreads = 128;        // 4 warps of 16 W rows
constexpr int kResSplits = 8;           // CTAs per head (cluster size)
constexpr int kResSteps = 4;            // 256-k stages per CTA (8192 / 256 / 8)
constexpr int kResSmemStages = 2;       // in shared memory (one TMA copy)
constexpr int kResRegStages = kResSteps - kResSmemStages;   // in registers
constexpr int kResChunks = 8;           // 32-k chunks per stage

struct ResLayout {
    uint32_t w, x, recv, full, recv_bar, abort_flag, total;
};

// owned: tokens per rank at most (ceil(mt / S))
__host__ __device__ inline ResLayout res_layout(int mt)
{
    ResLayout L;
    uint32_t off = 0;
    L.w = off;
    off += kResSmemStages * 4 * kBoxBytesW;
    L.x = off;
    off += kResSteps * 4 * (uint32_t)mt * 128;
    L.recv = off;   // [local token][source rank][64] FP32 partials
    off += (uint32_t)((mt + kResSplits - 1) / kResSplits) * kResSplits * kHeadDim * 4;
    L.full = off;
    off += 8;
    L.recv_bar = off;
    off += 8;
    L.abort_flag = off;
    off += 8;
    L.total = off;
    return L;
}

__host__ __device__ inline uint32_t res_smem_bytes(int mt) { return res_layout(mt).total + 1024; }

__device__ __forceinline__ void tma_load_4d_front(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0,
                                                  int c1, int c2, int c3, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
        : "memory");
}

// 16 bytes of W, streamed once: not kept in L1, first out of L2
__device__ __forceinline__ uint4 ldg_stream(const void *ptr, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr), "l"(policy));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
                 "r"(__float_as_uint(v)), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int MT>
__global__ void __launch_bounds__(kResThreads, 2)
    qkv_front_resident_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                              const FrontParams p)
{
    constexpr int NT = MT / 8;
    constexpr int kOwnedMax = (MT + kResSplits - 1) / kResSplits;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    const ResLayout L = res_layout(MT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int S = kResSplits;
    const uint32_t rank = cluster_rank();
    const int head = blockIdx.y;
    const uint32_t sW = smem_u32(smem + L.w), sX = smem_u32(smem + L.x), sRecv = smem_u32(smem + L.recv);
    const uint32_t full_bar = smem_u32(smem + L.full), recv_bar = smem_u32(smem + L.recv_bar);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.abort_flag);
    const int q_heads = kQPerKv * p.nkv;
    const int kind = head < q_heads ? kQ : head < q_heads + p.nkv ? kK : head < q_heads + 2 * p.nkv ? kV : kGate;
    // tokens this rank owns: u = rank + lt * S for lt < owned
    const int owned = (int)rank < p.M ? (p.M - 1 - (int)rank) / S + 1 : 0;
    const uint32_t smem_tx = kResSmemStages * 4 * kBoxBytesW + kResSteps * 4 * MT * 128;

    if (threadIdx.x == 0) {
        mbar_init(full_bar, 1);
        mbar_init(recv_bar, 1);
        *s_abort = 0;
        // the arrivals now, the bytes as they land (the partials from the
        // other ranks may complete before this CTA gets to its own wait)
        mbar_expect_tx(full_bar, smem_tx);
        mbar_expect_tx(recv_bar, (uint32_t)((S - 1) * owned * kHeadDim * 4));
        fence_barrier_init();
        griddep_launch_dependents();
    }
    __syncthreads();
    cluster_arrive_release();   // every rank's barriers are initialised before any st.async

    // ---- before the PDL wait: the weights (never written by a kernel in flight) ----
    const uint64_t pol_w = policy_evict_first();
    uint4 wr[kResRegStages][kResChunks][2];   // rows g and g + 8 of the warp's 16
    {
        const uint16_t *row0 = p.W + (size_t)(head * kHeadDim + warp * 16 + g) * kHidden + 8 * t;
#pragma unroll
        for (int i = 0; i < kResRegStages; ++i) {
            const int k0 = ((int)rank + (kResSmemStages + i) * S) * (kBoxK * 4);
#pragma unroll
            for (int c = 0; c < kResChunks; ++c) {
                wr[i][c][0] = ldg_stream(row0 + k0 + 32 * c, pol_w);
                wr[i][c][1] = ldg_stream(row0 + 8 * kHidden + k0 + 32 * c, pol_w);
            }
        }
    }
    // stages 0 and 1: 64 rows x 4 boxes x 2 stages in one copy, issued after
    // this thread's own register loads (issued before them, the copy was
    // measured to land about 1.5 us later per call at N = 1152)
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmX);
        tma_load_4d_front(sW, &tmW, full_bar, 0, head * kHeadDim, 4 * (int)rank, 0, pol_w);
    }

    griddep_wait();   // x, positions, slots, cos|sin come from the kernels before this one
    if (threadIdx.x == 0)
        tma_load_4d_front(sX, &tmX, full_bar, 0, 0, 4 * (int)rank, 0, policy_evict_last());

    // this warp's token (the finish: warp lt takes local token lt)
    const int u = (int)rank + warp * S;
    int flag = 0;
    int64_t slot = -1;
    float cs_c = 0.f, cs_s = 0.f;
    if (warp < owned) {
        const int64_t pos = p.positions[u];
        slot = p.slots[u];
        const bool pos_ok = pos >= 0 && pos < p.cos_rows;
        const bool slot_over = slot >= p.num_pages * (int64_t)kPageSlots;
        flag = (pos_ok ? 1 : 0) | (slot >= 0 && !slot_over && pos_ok ? 2 : 0);
        if (pos_ok && (kind == kQ || kind == kK)) {
            cs_c = p.cos_sin[pos * kHeadDim + lane];
            cs_s = p.cos_sin[pos * kHeadDim + 32 + lane];
        }
        if (head == 0 && lane == 0 && (!pos_ok || slot_over))
            atomicOr(&g_status, (pos_ok ? 0u : QKVF_STATUS_BAD_POSITION) | (slot_over ? QKVF_STATUS_BAD_SLOT : 0u));
    }

    // ---- contraction ---------------------------------------------------
    // Each step takes one shared-memory box (four k16 steps, ldmatrix) and
    // two register chunks (four k16 steps, W already in registers), so the
    // two instruction streams hide each other's latency.  One token tile:
    // eight independent accumulator chains (box steps 0..3, register steps
    // 4..7); two tiles: four chains per tile, shared by both streams.
    constexpr int kChains = NT == 1 ? 8 : 4;
    float acc[NT][kChains][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int kk = 0; kk < kChains; ++kk)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[nt][kk][r] = 0.f;
    const bool landed = mbar_try_wait(full_bar, 0) || bounded_wait(full_bar, 0, s_abort, p.wait_limit_ns, true);
    if (__all_sync(0xffffffffu, landed)) {
        const uint32_t a_row = (uint32_t)(warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8);
        const uint32_t a_off = a_row * 128u, a_hi = (uint32_t)(lane >> 4);
        const uint32_t b_tok = NT == 2 ? (uint32_t)((lane & 7) + ((lane >> 4) << 3)) : (uint32_t)(lane & 7);
        const uint32_t b_off = b_tok * 128u, b_hi = (uint32_t)((lane >> 3) & 1);
        const uint32_t sw = (uint32_t)(lane & 7);
        constexpr int kBoxes = kResSmemStages * 4;                        // 8
        constexpr int kRegChunksPerBox = kResRegStages * kResChunks / kBoxes;   // 2
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) {
            // shared-memory box bx: ldmatrix from the 128-byte swizzled rows
            const uint32_t wbox = sW + (uint32_t)bx * kBoxBytesW;
            const uint32_t xbox = sX + (uint32_t)bx * (MT * 128);
            uint32_t a[4][4], bb[4][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                ldsm_x4(wbox + a_off + ((((uint32_t)(2 * kk) + a_hi) ^ sw) << 4), a[kk][0], a[kk][1], a[kk][2],
                        a[kk][3]);
                const uint32_t baddr = xbox + b_off + ((((uint32_t)(2 * kk) + b_hi) ^ sw) << 4);
                if constexpr (NT == 2)
                    ldsm_x4(baddr, bb[kk][0], bb[kk][1], bb[kk][2], bb[kk][3]);
                else
                    ldsm_x2(baddr, bb[kk][0], bb[kk][1]);
            }
            // register chunks: x in the same k order, 16 bytes per lane from the box
            uint4 xv[kRegChunksPerBox][NT];
#pragma unroll
            for (int q = 0; q < kRegChunksPerBox; ++q) {
                const int rc = bx * kRegChunksPerBox + q, i = rc / kResChunks, c = rc % kResChunks;
                const uint32_t xrb = sX + (uint32_t)((kResSmemStages + i) * 4 + c / 2) * (MT * 128);
                const uint32_t chunk = (uint32_t)(4 * (c & 1) + t);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {   // token row nt 8 + g: swizzle phase g
                    // rows past M hold zeros: only lanes of real tokens read
                    xv[q][nt] = make_uint4(0u, 0u, 0u, 0u);
                    if (nt * 8 + g < p.M)
                        xv[q][nt] = lds128(xrb + (uint32_t)(nt * 8 + g) * 128u + ((chunk ^ (uint32_t)g) << 4));
                }
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16_16816(acc[0][kk], a[kk][0], a[kk][1], a[kk][2], a[kk][3], bb[kk][0], bb[kk][1]);
                if constexpr (NT == 2)
                    mma_bf16_16816(acc[1][kk], a[kk][0], a[kk][1], a[kk][2], a[kk][3], bb[kk][2], bb[kk][3]);
            }
#pragma unroll
            for (int q = 0; q < kRegChunksPerBox; ++q) {
                const int rc = bx * kRegChunksPerBox + q, i = rc / kResChunks, c = rc % kResChunks;
                const uint4 wg = wr[i][c][0], wg8 = wr[i][c][1];
                constexpr int base = NT == 1 ? 4 : 0;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_bf16_16816(acc[nt][base + ((2 * q) & 3)], wg.x, wg8.x, wg.y, wg8.y, xv[q][nt].x, xv[q][nt].y);
                    mma_bf16_16816(acc[nt][base + ((2 * q + 1) & 3)], wg.z, wg8.z, wg.w, wg8.w, xv[q][nt].z,
                                   xv[q][nt].w);
                }
            }
        }
    }
    float sum[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float v = __fadd_rn(__fadd_rn(acc[nt][0][r], acc[nt][1][r]), __fadd_rn(acc[nt][2][r], acc[nt][3][r]));
            if constexpr (kChains == 8)
                v = __fadd_rn(v, __fadd_rn(__fadd_rn(acc[nt][4][r], acc[nt][5][r]),
                                           __fadd_rn(acc[nt][6][r], acc[nt][7][r])));
            sum[nt][r] = v;
        }

    // ---- send: token tok's rows to rank tok % S, slot [tok / S][rank][row] ----
    cluster_wait_acquire();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + 2 * t + (e & 1);
            const int row = warp * 16 + g + ((e >> 1) << 3);
            if (tok < p.M) {
                const uint32_t owner = (uint32_t)(tok % S);
                const uint32_t off = (uint32_t)((((tok / S) * S + (int)rank) * kHeadDim + row) * 4);
                if (owner == rank)
                    *reinterpret_cast<float *>(smem + L.recv + off) = sum[nt][e];
                else
                    st_async_f32(map_to_rank(sRecv + off, owner), sum[nt][e], map_to_rank(recv_bar, owner));
            }
        }
    if (owned == 0) {
        if (threadIdx.x == 0 && *s_abort)   // the copies into this CTA land before it leaves
            bounded_wait(full_bar, 0, s_abort, p.wait_limit_ns, false);
        return;   // nothing is read from this CTA's shared memory
    }
    __syncthreads();   // this rank's own partials are in its slots
    const bool got = mbar_try_wait(recv_bar, 0) || bounded_wait(recv_bar, 0, s_abort, p.wait_limit_ns, false);
    if (threadIdx.x == 0 && *s_abort) bounded_wait(full_bar, 0, s_abort, p.wait_limit_ns, false);

    // ---- finish: rank-order sum, round, norm, RoPE, store, insert ----------
    if (warp < owned && __all_sync(0xffffffffu, got)) {
        const float *part = reinterpret_cast<const float *>(smem + L.recv) + (size_t)warp * S * kHeadDim;
        float2 v = reinterpret_cast<const float2 *>(part)[lane];
#pragma unroll
        for (int src = 1; src < S; ++src) {
            const float2 w = reinterpret_cast<const float2 *>(part + src * kHeadDim)[lane];
            v.x = __fadd_rn(v.x, w.x);
            v.y = __fadd_rn(v.y, w.y);
        }
        finish_pair(p, head, kind, u, lane, v, flag, cs_c, cs_s, slot);
    }
    (void)kOwnedMax;
}

// One CTA waits on a barrier that nothing completes, through the front's own
// bounded wait; it must give up after limit_ns and raise the status bit.
__global__ void wait_selftest_kernel(unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        bounded_wait(smem_u32(&bar), 0u, reinterpret_cast<volatile int *>(&abort_flag), limit_ns,
                     false);
}

// ---- host side -------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool probed = false;
    bool ok = false;
    bool prepared = false;
    int sms = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
unsigned long long g_wait_limit_ns = 2000000000ull;
bool g_pdl = true;   // launch with programmatic stream serialization

using KernelFn = void (*)(CUtensorMap, CUtensorMap, FrontParams);

KernelFn kernel_for(int mt, bool tc)
{
    if (tc) return mt == 8 ? (KernelFn)qkv_front_kernel<8, true> : (KernelFn)qkv_front_kernel<16, true>;
    return mt == 8 ? (KernelFn)qkv_front_kernel<8, false> : (KernelFn)qkv_front_kernel<16, false>;
}
constexpr int kDefaultKB = 4;          // 64-k boxes per ring stage: 256 k, 32 KB of W
constexpr int kDefaultL2Prefetch = 3;  // W stages prefetched into L2 before the PDL wait
constexpr bool kDefaultTC = false;     // consumer: tcgen05 (true) or mma.sync

bool prepare_epi_kernel();
bool prepare_attn2_kernel();

int probe_device(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QKVF_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QKVF_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return QKVF_ERR_CUDA;
        d.probed = true;
        d.ok = (major == 10 && minor == 3);
        d.sms = sms;
    }
    if (!d.ok) return QKVF_ERR_DEVICE;
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return QKVF_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (!d.prepared) {
        for (int i = 0; i < 4; ++i) {
            KernelFn k = kernel_for(i & 1 ? 16 : 8, i >= 2);
            if (cudaFuncSetAttribute((const void *)k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmemPerCta) != cudaSuccess ||
                cudaFuncSetAttribute((const void *)k,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
                return QKVF_ERR_CUDA;
        }
        const void *res[2] = {(const void *)qkv_front_resident_kernel<8>, (const void *)qkv_front_resident_kernel<16>};
        for (int i = 0; i < 2; ++i)
            if (cudaFuncSetAttribute(res[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)res_smem_bytes(i ? 16 : 8)) != cudaSuccess)
                return QKVF_ERR_CUDA;
        if (!prepare_epi_kernel() || !prepare_attn2_kernel()) return QKVF_ERR_CUDA;
        d.prepared = true;
    }
    *out = &d;
    return QKVF_OK;
}

struct Variant {
    int mt, splits, stages, kb, l2_prefetch;
    bool tc;         // tcgen05 consumer (else mma.sync)
    bool resident;   // the resident engine: the CTA's whole W share on chip before the wait
};

int max_stages(int mt, int kb, int per_sm)
{
    const int budget = per_sm <= 1 ? kMaxSmemPerCta : kSmemPerSm / per_sm - kSmemReservedPerCta;
    int st = 2;
    while ((int)smem_bytes(mt, kb, st + 1) <= budget) ++st;
    return st;
}

// The launch shape for N columns and M tokens on `sms` SMs.  splits: the
// largest power of two (<= 16) that keeps heads x splits within the SM count;
// stages: as deep as shared memory allows, with one CTA per SM when each
// head is one CTA and two per SM for clusters (so that a GPC holds whole
// clusters), and no deeper than the CTA's number of K stages.  A split of 8
// leaves each CTA 128 KB of W, which the resident engine holds on chip.
Variant choose_variant(int N, int M, int sms)
{
    Variant v;
    const int heads = N / kHeadDim;
    v.mt = M <= 8 ? 8 : 16;
    v.kb = kDefaultKB;
    v.l2_prefetch = kDefaultL2Prefetch;
    v.tc = kDefaultTC;
    v.resident = false;
    v.splits = 1;
    while (v.splits < 16 && heads * v.splits * 2 <= sms) v.splits *= 2;
    if (v.splits == kResSplits && v.kb * kResSplits * kResSteps == kHidden / kBoxK) {
        v.resident = true;
        v.stages = kResSteps;
        return v;
    }
    const int per_sm = v.splits > 1 ? 2 : 1;
    const int steps = kHidden / (kBoxK * v.kb) / v.splits;
    v.stages = max_stages(v.mt, v.kb, per_sm);
    if (v.stages > steps) v.stages = steps;
    if (v.stages < 2) v.stages = 2;
    return v;
}

// Whether a variant can run: a power-of-two split and stage size that divide
// the 128 boxes of K, and a ring that fits the shared-memory limit.
bool variant_ok(const Variant &v)
{
    if (v.resident)   // fixed shape: 8 CTAs per head, 4 stages of 4 boxes
        return !v.tc && v.splits == kResSplits && v.kb * kResSplits * kResSteps == kHidden / kBoxK &&
               v.stages == kResSteps;
    const bool pow2_s = v.splits == 1 || v.splits == 2 || v.splits == 4 || v.splits == 8 ||
                        v.splits == 16;
    const bool kb_ok = v.kb == 1 || v.kb == 2 || v.kb == 4;
    if (!pow2_s || !kb_ok || v.stages < 2 || v.l2_prefetch < 0 || v.l2_prefetch > 64) return false;
    if (v.splits * v.kb > kHidden / kBoxK) return false;
    return (int)smem_bytes(v.mt, v.kb, v.stages) <= kMaxSmemPerCta;
}

bool aligned(const void *ptr, uintptr_t a) { return ((uintptr_t)ptr % a) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return na && nb && x < y + nb && y < x + na;
}

const char *check_args(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                       const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows,
                       uint16_t *out, uint16_t *kv_cache, int64_t num_pages, int M, int N,
                       int num_kv_heads, int *code)
{
    *code = QKVF_ERR_TOKENS;
    if (M < 0 || M > kMaxTokens) return "M must be 0..16 tokens";
    *code = QKVF_ERR_SHAPE;
    if (num_kv_heads < 1 || num_kv_heads > 64)
        return "num_kv_heads must be 1..64";
    if (N != 2 * (kQPerKv + 1) * kHeadDim * num_kv_heads)
        return "N must be 1152 * num_kv_heads: rows [q | k | v | gate], 8 q and 8 gate heads of 64 per KV head";
    *code = QKVF_ERR_SIZES;
    if (cos_sin_rows < 1 || cos_sin_rows > (int64_t(1) << 40)) return "cos_sin_rows must be >= 1";
    if (num_pages < 1 || num_pages > (int64_t(1) << 36)) return "num_pages must be >= 1";
    if (M == 0) {
        *code = QKVF_OK;
        return nullptr;
    }
    *code = QKVF_ERR_NULL;
    if (!x || !W || !positions || !slots || !cos_sin || !out || !kv_cache)
        return "a required pointer is NULL";
    *code = QKVF_ERR_ALIGN;
    if (!aligned(x, 16) || !aligned(W, 16))
        return "x and W must be 16-byte aligned bf16 [rows, 8192]";
    if (!aligned(out, 16) || !aligned(kv_cache, 16) || !aligned(cos_sin, 16))
        return "out, kv_cache and cos_sin must be 16-byte aligned";
    if (!aligned(positions, 8) || !aligned(slots, 8))
        return "positions and slots must be 8-byte aligned int64";
    *code = QKVF_ERR_ARG;
    const size_t out_b = (size_t)M * N * 2;
    const size_t cache_b = (size_t)num_pages * num_kv_heads * kPageSlots * kSlotWidth * 2;
    const size_t x_b = (size_t)M * kHidden * 2, w_b = (size_t)N * kHidden * 2;
    const size_t cs_b = (size_t)cos_sin_rows * kHeadDim * 4, idx_b = (size_t)M * 8;
    const void *ins[] = {x, W, cos_sin, positions, slots};
    const size_t in_b[] = {x_b, w_b, cs_b, idx_b, idx_b};
    for (int i = 0; i < 5; ++i)
        if (overlap(ins[i], in_b[i], out, out_b) || overlap(ins[i], in_b[i], kv_cache, cache_b))
            return "an input overlaps out or kv_cache";
    if (overlap(out, out_b, kv_cache, cache_b)) return "out overlaps kv_cache";
    *code = QKVF_OK;
    return nullptr;
}

// The ring's maps: W and x viewed as 3-D (64 k within a block, rows, the
// 128 blocks of 64 k, 128 bytes apart), so that one box of kb blocks is a
// whole ring stage; each block lands as 64 (W) or mt (x) rows of 128
// swizzled bytes, block after block.
int encode_maps(const uint16_t *x, const uint16_t *W, int M, int N, int mt, int kb, CUtensorMap *mw,
                CUtensorMap *mx)
{
    const cuuint64_t stride[2] = {(cuuint64_t)kHidden * 2, 128};
    const cuuint32_t estride[3] = {1, 1, 1};
    const cuuint64_t wdim[3] = {(cuuint64_t)kBoxK, (cuuint64_t)N, (cuuint64_t)(kHidden / kBoxK)};
    const cuuint32_t wbox[3] = {(cuuint32_t)kBoxK, (cuuint32_t)kHeadDim, (cuuint32_t)kb};
    if (g_encode(mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void *)W, wdim, stride, wbox, estride,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QKVF_ERR_CUDA;
    // x rows past M read as zeros (out-of-bounds fill), so a tile of 8 or 16
    // tokens covers any M
    const cuuint64_t xdim[3] = {(cuuint64_t)kBoxK, (cuuint64_t)M, (cuuint64_t)(kHidden / kBoxK)};
    const cuuint32_t xbox[3] = {(cuuint32_t)kBoxK, (cuuint32_t)mt, (cuuint32_t)kb};
    if (g_encode(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void *)x, xdim, stride, xbox, estride,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QKVF_ERR_CUDA;
    return QKVF_OK;
}

// The resident engine's maps: W and x viewed as 4-D (64 k, rows, 4S blocks of
// 64 k with a stride of 128 bytes, the CTA's stages 512 S bytes apart), so
// that one box is a CTA's whole stripe of stages (x) or its first two (W).
int encode_resident_maps(const uint16_t *x, const uint16_t *W, int M, int N, int mt, CUtensorMap *mw,
                         CUtensorMap *mx)
{
    const int S = kResSplits;
    const cuuint64_t stride[3] = {(cuuint64_t)kHidden * 2, 128, (cuuint64_t)512 * S};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    const cuuint64_t wdim[4] = {(cuuint64_t)kBoxK, (cuuint64_t)N, (cuuint64_t)4 * S, (cuuint64_t)kResSteps};
    const cuuint32_t wbox[4] = {(cuuint32_t)kBoxK, (cuuint32_t)kHeadDim, 4, (cuuint32_t)kResSmemStages};
    if (g_encode(mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void *)W, wdim, stride, wbox, estride,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QKVF_ERR_CUDA;
    // rows past M read as zeros
    const cuuint64_t xdim[4] = {(cuuint64_t)kBoxK, (cuuint64_t)M, (cuuint64_t)4 * S, (cuuint64_t)kResSteps};
    const cuuint32_t xbox[4] = {(cuuint32_t)kBoxK, (cuuint32_t)mt, 4, (cuuint32_t)kResSteps};
    if (g_encode(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void *)x, xdim, stride, xbox, estride,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return QKVF_ERR_CUDA;
    return QKVF_OK;
}

int launch_front(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                 const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows, uint16_t *out,
                 uint16_t *kv_cache, int64_t num_pages, int M, int N, int num_kv_heads,
                 const Variant &v, void *stream)
{
    CUtensorMap mw, mx;
    int rc = v.resident ? encode_resident_maps(x, W, M, N, v.mt, &mw, &mx)
                        : encode_maps(x, W, M, N, v.mt, v.kb, &mw, &mx);
    if (rc != QKVF_OK) return rc;
    FrontParams prm;
    prm.W = W;
    prm.positions = positions;
    prm.slots = slots;
    prm.cos_sin = cos_sin;
    prm.out = out;
    prm.kv_cache = kv_cache;
    prm.cos_rows = cos_sin_rows;
    prm.num_pages = num_pages;
    prm.wait_limit_ns = g_wait_limit_ns;
    prm.M = M;
    prm.N = N;
    prm.nkv = num_kv_heads;
    prm.splits = v.splits;
    prm.stages = v.stages;
    prm.kb = v.kb;
    prm.l2_prefetch = v.l2_prefetch;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)v.splits, (unsigned)(N / kHeadDim), 1);
    cfg.blockDim = dim3(v.resident ? kResThreads : kThreads, 1, 1);
    cfg.dynamicSmemBytes = v.resident ? res_smem_bytes(v.mt) : smem_bytes(v.mt, v.kb, v.stages);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attrs[3];
    int na = 0;
    if (v.splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)v.splits;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
        // a cluster's CTAs on distinct SMs where possible: two CTAs of one
        // call on one SM share its shared-memory path and tensor pipes
        attrs[na].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
        attrs[na].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicySpread;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    const KernelFn k = v.resident ? (v.mt == 8 ? (KernelFn)qkv_front_resident_kernel<8>
                                               : (KernelFn)qkv_front_resident_kernel<16>)
                                  : kernel_for(v.mt, v.tc);
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, mw, mx, prm);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QKVF_ERR_CUDA;
    }
    return QKVF_OK;
}

}  // namespace qkvf

#include "qknorm_rope_kv_insert.cuh"
#include "layer_front.cuh"
#include "attn2.cuh"

using namespace qkvf;

extern "C" {

const char *qkv_front_strerror(int code)
{
    switch (code) {
    case QKVF_OK: return "ok";
    case QKVF_ERR_TOKENS: return "M must be 0..16 tokens";
    case QKVF_ERR_SHAPE: return "N must be 1152 * num_kv_heads with num_kv_heads >= 1";
    case QKVF_ERR_NULL: return "a required pointer is NULL";
    case QKVF_ERR_ALIGN: return "a pointer is not aligned (16 bytes; 8 for positions and slots)";
    case QKVF_ERR_DEVICE: return "the current GPU is not compute capability 10.3 (sm_103a)";
    case QKVF_ERR_CUDA: return "a CUDA call failed";
    case QKVF_ERR_SIZES: return "cos_sin_rows and num_pages must be >= 1";
    case QKVF_ERR_VARIANT: return "this variant cannot run this shape";
    case QKVF_ERR_ARG: return "bad argument (overlapping buffers or out-of-range setting)";
    default: return "unknown qkv_front error";
    }
}

const char *qkv_front_unsupported(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                                  const int64_t *slots, const float *cos_sin,
                                  int64_t cos_sin_rows, uint16_t *out, uint16_t *kv_cache,
                                  int64_t num_pages, int M, int N, int num_kv_heads)
{
    int code;
    const char *why = check_args(x, W, positions, slots, cos_sin, cos_sin_rows, out, kv_cache,
                                 num_pages, M, N, num_kv_heads, &code);
    if (why) return why;
    DeviceState *d;
    int rc = probe_device(&d);
    if (rc != QKVF_OK) return qkv_front_strerror(rc);
    return nullptr;
}

int qkv_front_launch(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                     const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows,
                     uint16_t *out, uint16_t *kv_cache, int64_t num_pages, int M, int N,
                     int num_kv_heads, void *stream)
{
    if (M == 0) return QKVF_OK;
    DeviceState *d;
    int rc = probe_device(&d);
    if (rc != QKVF_OK) return rc;
    const Variant v = choose_variant(N, M, d->sms);
    return launch_front(x, W, positions, slots, cos_sin, cos_sin_rows, out, kv_cache, num_pages, M,
                        N, num_kv_heads, v, stream);
}

int qkv_front(const uint16_t *x, const uint16_t *W, const int64_t *positions,
              const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows, uint16_t *out,
              uint16_t *kv_cache, int64_t num_pages, int M, int N, int num_kv_heads, void *stream)
{
    int code;
    if (check_args(x, W, positions, slots, cos_sin, cos_sin_rows, out, kv_cache, num_pages, M, N,
                   num_kv_heads, &code))
        return code;
    return qkv_front_launch(x, W, positions, slots, cos_sin, cos_sin_rows, out, kv_cache,
                            num_pages, M, N, num_kv_heads, stream);
}

int qkv_front_variant(int N, int M, int *tiles, int *stages, int *splits, int *kb, int *consumer)
{
    if (M < 1 || M > kMaxTokens) return QKVF_ERR_TOKENS;
    if (N < 1152 || N % 1152) return QKVF_ERR_SHAPE;
    DeviceState *d;
    int rc = probe_device(&d);
    if (rc != QKVF_OK) return rc;
    const Variant v = choose_variant(N, M, d->sms);
    if (tiles) *tiles = v.mt / 8;
    if (stages) *stages = v.stages;
    if (splits) *splits = v.splits;
    if (kb) *kb = v.kb;
    if (consumer)
        *consumer = v.resident ? QKVF_CONSUMER_RESIDENT : v.tc ? QKVF_CONSUMER_TCGEN05 : QKVF_CONSUMER_MMA_SYNC;
    return QKVF_OK;
}

int qkv_front_launch_variant(const uint16_t *x, const uint16_t *W, const int64_t *positions,
                             const int64_t *slots, const float *cos_sin, int64_t cos_sin_rows,
                             uint16_t *out, uint16_t *kv_cache, int64_t num_pages, int M, int N,
                             int num_kv_heads, int splits, int stages, int kb, int consumer,
                             void *stream)
{
    int code;
    if (check_args(x, W, positions, slots, cos_sin, cos_sin_rows, out, kv_cache, num_pages, M, N,
                   num_kv_heads, &code))
        return code;
    if (M == 0) return QKVF_OK;
    if (consumer != QKVF_CONSUMER_DEFAULT && consumer != QKVF_CONSUMER_MMA_SYNC &&
        consumer != QKVF_CONSUMER_TCGEN05 && consumer != QKVF_CONSUMER_RESIDENT)
        return QKVF_ERR_VARIANT;
    Variant v;
    v.mt = M <= 8 ? 8 : 16;
    v.splits = splits;
    v.stages = stages;
    v.kb = kb == 0 ? kDefaultKB : kb;
    v.l2_prefetch = kDefaultL2Prefetch;
    v.tc = consumer == QKVF_CONSUMER_DEFAULT ? kDefaultTC : consumer == QKVF_CONSUMER_TCGEN05;
    v.resident = consumer == QKVF_CONSUMER_RESIDENT;
    if (!variant_ok(v)) return QKVF_ERR_VARIANT;
    DeviceState *d;
    int rc = probe_device(&d);
    if (rc != QKVF_OK) return rc;
    return launch_front(x, W, positions, slots, cos_sin, cos_sin_rows, out, kv_cache, num_pages, M,
                        N, num_kv_heads, v, stream);
}

int qkv_front_prepare(int N, int num_kv_heads)
{
    if (num_kv_heads < 1 || N != 2 * (kQPerKv + 1) * kHeadDim * num_kv_heads) return QKVF_ERR_SHAPE;
    DeviceState *d;
    return probe_device(&d);
}

int qkv_front_status(unsigned int *bits)
{
    if (!bits) return QKVF_ERR_NULL;
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return QKVF_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return QKVF_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) return QKVF_ERR_CUDA;
    *bits = v;
    return QKVF_OK;
}

// Copies a call's host inputs into the staging buffer from the GPU itself,
// for pinned (device-mapped) host memory: x as 16-byte loads, positions and
// slots by the first M threads.  The host reads are issued before the wait
// for the kernel before (whose front may still read the staging buffer);
// the stores after it.  Launched with PDL, and it lets the front launch at
// once, so the front's weight stream starts while x is still arriving.
constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads) stage_from_host_kernel(
    const uint4 *x_host, const int64_t *pos_host, const int64_t *slot_host, uint4 *x, int64_t *pos,
    int64_t *slot, int n16, int M)
{
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int i = blockIdx.x * kStageThreads + threadIdx.x;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (i < n16) v = __ldcv(x_host + i);   // not cached: the host rewrites it between calls
    int64_t pv = 0, sv = 0;
    if (i < M) {
        pv = __ldcv(reinterpret_cast<const long long *>(pos_host) + i);
        sv = __ldcv(reinterpret_cast<const long long *>(slot_host) + i);
    }
    griddep_wait();
    if (i < n16) x[i] = v;
    if (i < M) {
        pos[i] = pv;
        slot[i] = sv;
    }
}

// The device address of a pinned (page-locked, device-mapped) host buffer,
// or null when the GPU cannot reach it (pageable memory: copy it instead).
static void *mapped_host(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// staging layout of qkv_front_from_host: x | positions | slots | out, each
// starting on a 256-byte boundary
struct Staging {
    uint64_t x, pos, slot, out, total;
};

static Staging staging_layout(int M, int N)
{
    auto up = [](uint64_t v) { return (v + 255u) & ~(uint64_t)255u; };
    Staging st;
    st.x = 0;
    st.pos = up(st.x + (uint64_t)M * kHidden * 2);
    st.slot = up(st.pos + (uint64_t)M * 8);
    st.out = up(st.slot + (uint64_t)M * 8);
    st.total = up(st.out + (uint64_t)M * N * 2);
    return st;
}

uint64_t qkv_front_staging_bytes(int M, int N)
{
    if (M < 0 || M > kMaxTokens || N < 0) return 0;
    return staging_layout(M, N).total;
}

int qkv_front_from_host(const uint16_t *x_host, const int64_t *positions_host,
                        const int64_t *slots_host, uint16_t *out_host, const uint16_t *W,
                        const float *cos_sin, int64_t cos_sin_rows, uint16_t *kv_cache,
                        int64_t num_pages, void *staging, uint64_t staging_bytes, int M, int N,
                        int num_kv_heads, void *stream)
{
    if (M < 0 || M > kMaxTokens) return QKVF_ERR_TOKENS;
    if (M == 0) return QKVF_OK;
    if (!x_host || !positions_host || !slots_host || !out_host || !staging) return QKVF_ERR_NULL;
    if ((uintptr_t)staging % 256) return QKVF_ERR_ALIGN;
    const Staging st = staging_layout(M, N);
    if (staging_bytes < st.total) return QKVF_ERR_SIZES;
    uint8_t *base = static_cast<uint8_t *>(staging);
    const uint16_t *x = reinterpret_cast<const uint16_t *>(base + st.x);
    const int64_t *pos = reinterpret_cast<const int64_t *>(base + st.pos);
    const int64_t *slots = reinterpret_cast<const int64_t *>(base + st.slot);
    uint16_t *out = reinterpret_cast<uint16_t *>(base + st.out);
    int code;
    if (check_args(x, W, pos, slots, cos_sin, cos_sin_rows, out, kv_cache, num_pages, M, N,
                   num_kv_heads, &code))
        return code;
    const cudaStream_t s = (cudaStream_t)stream;
    DeviceState *d;
    int rc = probe_device(&d);
    if (rc != QKVF_OK) return rc;
    // pinned host buffers are read and written by the kernels over the
    // host link; pageable ones go through copies on the stream
    const void *xm = mapped_host(x_host), *pm = mapped_host(positions_host), *sm = mapped_host(slots_host);
    void *om = mapped_host(out_host);
    if (xm && pm && sm && (uintptr_t)xm % 16 == 0) {
        const int n16 = M * kHidden * 2 / 16;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((n16 + kStageThreads - 1) / kStageThreads), 1, 1);
        cfg.blockDim = dim3(kStageThreads, 1, 1);
        cfg.stream = s;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, stage_from_host_kernel, static_cast<const uint4 *>(xm),
                               static_cast<const int64_t *>(pm), static_cast<const int64_t *>(sm),
                               reinterpret_cast<uint4 *>(const_cast<uint16_t *>(x)), const_cast<int64_t *>(pos),
                               const_cast<int64_t *>(slots), n16, M) != cudaSuccess) {
            (void)cudaGetLastError();
            return QKVF_ERR_CUDA;
        }
    } else if (cudaMemcpyAsync((void *)x, x_host, (size_t)M * kHidden * 2, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess ||
               cudaMemcpyAsync((void *)pos, positions_host, (size_t)M * 8, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess ||
               cudaMemcpyAsync((void *)slots, slots_host, (size_t)M * 8, cudaMemcpyHostToDevice, s) !=
                   cudaSuccess) {
        return QKVF_ERR_CUDA;
    }
    const bool out_direct = om && (uintptr_t)om % 16 == 0;
    rc = qkv_front_launch(x, W, pos, slots, cos_sin, cos_sin_rows,
                          out_direct ? static_cast<uint16_t *>(om) : out, kv_cache, num_pages, M, N,
                          num_kv_heads, stream);
    if (rc != QKVF_OK) return rc;
    if (!out_direct &&
        cudaMemcpyAsync(out_host, out, (size_t)M * N * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QKVF_ERR_CUDA;
    return QKVF_OK;
}

int qkv_front_selftest_wait(int64_t timeout_ns, void *stream)
{
    if (timeout_ns < 1 || timeout_ns > 1000000000ll) return QKVF_ERR_ARG;
    DeviceState *d;
    int rc = probe_device(&d);
    if (rc != QKVF_OK) return rc;
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((unsigned long long)timeout_ns);
    return cudaGetLastError() == cudaSuccess ? QKVF_OK : QKVF_ERR_CUDA;
}

int qkv_front_set_pdl(int enable)
{
    if (enable != 0 && enable != 1) return QKVF_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_pdl = enable != 0;
    return QKVF_OK;
}

int qkv_front_set_wait_limit(int64_t ns)
{
    if (ns < 1000 || ns > 10000000000ll) return QKVF_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_wait_limit_ns = (unsigned long long)ns;
    return QKVF_OK;
}

}  // extern "C"

// ---- attn2 split-KV without a caller's workspace ---------------------------
//
// For callers that cannot allocate device memory themselves: a plugin whose
// host process owns every device allocation through its own pool, or a
// decode step that must not risk cudaMalloc's implicit synchronisation or a
// failed allocation halfway through.  Their split-KV partials go to one
// file-scope array that every GPU loading this library holds until exit
// (256 slots of 17152 bytes, 4.39 MB).  The engine reads no slot it has not
// written in the same call, so the array needs no clearing between calls;
// calls that overlap on the GPU share it and race.

namespace qkvf {

constexpr int kNoAllocSlots = 256;
constexpr size_t kNoAllocBytes = (size_t)kNoAllocSlots * kA2WsSlotFloats * 4;
static __device__ __align__(256) float g_a2_noalloc_scratch[(size_t)kNoAllocSlots * kA2WsSlotFloats];

// The array's device address in the current context (host code only sees a
// stand-in under its name).  Looked up on every call: a cached address
// would outlive a device reset, after which the module is loaded anew.
int noalloc_scratch(void **ptr)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_a2_noalloc_scratch) != cudaSuccess || !p) {
        (void)cudaGetLastError();
        return QKVF_ERR_CUDA;
    }
    *ptr = p;
    return QKVF_OK;
}

}  // namespace qkvf

extern "C" {

int attn2_split_kv_noalloc(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                           const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                           int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                           uint16_t *out, int splits, void *stream)
{
    int code;
    if (qkvf::check_attn2_args(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                               num_reqs, N, num_kv_heads, window, scale, eps, out, &code))
        return code;
    if (splits < 0 || splits > qkvf::kA2WsMaxSplits) return QKVF_ERR_VARIANT;
    if (num_reqs == 0) return QKVF_OK;
    // one split writes no partials: only splits > 1 use the array's slots
    if (splits > 1 && (int64_t)num_reqs * num_kv_heads * splits > qkvf::kNoAllocSlots)
        return QKVF_ERR_SIZES;   // more partial slots than the array holds
    qkvf::DeviceState *d;
    int rc = qkvf::probe_device(&d);
    if (rc != QKVF_OK) return rc;
    if (splits == 0)
        splits = qkvf::attn2_split_kv_splits_for(num_reqs, num_kv_heads, max_blocks, window, d->sms);
    if (splits == 1)   // the direct path: each CTA finishes its own rows, no scratch
        return qkvf::launch_attn2(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                                  num_reqs, N, num_kv_heads, window, scale, eps, out, 1, nullptr, d->sms,
                                  stream);
    if ((int64_t)num_reqs * num_kv_heads * splits > qkvf::kNoAllocSlots) return QKVF_ERR_SIZES;
    void *scratch = nullptr;
    rc = qkvf::noalloc_scratch(&scratch);
    if (rc != QKVF_OK) return rc;
    return attn2_split_kv(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens, num_reqs, N,
                          num_kv_heads, window, scale, eps, out, splits, scratch, qkvf::kNoAllocBytes,
                          stream);
}

}  // extern "C"
