// attn2: the consumer of the paged cache the front fills — decode attention of
// the 8-token verify step fused with the output's weightless RMS norm and
// sigmoid gate (included by qkv_front.cu: one translation unit).
//
// Source: page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.
// cute_ops", attn2 paragraph: one request = 1 + 7 draft tokens = 8 query rows,
// head_dim 64, 8 query heads per KV head, the bf16 cache [pages, num_kv_heads,
// 16, 128] (K | V per slot), any context length L >= 8, an optional sliding
// window, one launch for the rank's KV heads; the result is the o_proj input.
// Readings where the page is silent (the same in the oracle): row i of a
// request is the token at position L - 8 + i and sees keys j <= L - 8 + i
// (and j > L - 8 + i - W with a window W); key j is slot j % 16 of page
// block_table[r][j / 16]; q head h reads KV head h / 8 and is gated by gate
// head h of its row; out = bf16(o / sqrt(mean(o^2) + eps) * sigmoid(gate))
// with o = softmax(scale q K^T) V.
//
// Design: a CTA per (request r, KV head g, split z).  A producer warp streams
// the CTA's pages (p0 + z, p0 + z + S, ...) into a ring of blocks of 4 pages
// (one 4-KB TMA box per page, 128-byte swizzled: K rows of slots 0-7, V rows
// of slots 0-7, K rows of slots 8-15, V rows of slots 8-15, 1 KB each)
// sharing one full / empty barrier pair.  Groups of four compute warps (16 of
// the 64 query rows each — 8 tokens x 8 heads, row 8 i + j) take blocks of 4
// pages in turn: one thread of the group issues Q K^T for the block's 64 keys
// as four tcgen05.mma (M = 64 rows, N = 64 keys, K = 16; the keys' 8-row
// groups 2 KB apart) into the group's 64 tensor-memory columns, the warps
// read the scores back with tcgen05.ld in the mma.sync accumulator layout,
// run the online softmax (base 2; masks only near the causal / window edges)
// and P V with mma.sync, P going from the score registers straight into the
// A fragments.  Each group keeps its own (max, sum, O), folded into one per
// CTA in group order.  Two shapes of the kernel (A2Shape): 3 groups and a
// 12-block ring, one CTA per SM; 2 groups and a 4-block ring, two CTAs per
// SM, for a direct launch with more (request, KV head) pairs than SMs.
// Cluster engine: the S CTAs of a (request, KV head) form a cluster and merge
// their partials through distributed shared memory in rank order — no global
// workspace, deterministic for a launch shape — then each rank finishes 64 / S
// rows: o-norm, gate, BF16 store.  Split-KV engine: no cluster; the partials
// go to a caller's workspace and a second grid merges them.

namespace qkvf {

constexpr int kA2Block = 4;                               // pages per softmax step (16 per page)
constexpr uint32_t kA2PageBytes = 4096;                   // one box: K 0-7, V 0-7, K 8-15, V 8-15
static_assert(32 % kA2Block == 0, "a block's table entries lie in one 32-entry chunk");

// The kernel's two shapes, by its groups of 4 compute warps (plus one
// producer warp): 3 groups, a 12-block ring (192 KB) and one CTA per SM, the
// default; 2 groups, a 4-block ring (64 KB) and two CTAs per SM, for a direct
// launch whose (request, KV head) pairs outnumber the SMs (all of its CTAs in
// one wave, 4 block chains per SM).
template <int kG>
struct A2Shape {
    static constexpr int groups = kG;
    static constexpr int compute_warps = 4 * kG;
    static constexpr int threads = 32 * (compute_warps + 1);   // the last warp produces
    static constexpr int ring_blocks = kG == 3 ? 12 : 4;
    static constexpr int ctas_per_sm = kG == 3 ? 1 : 2;
    static constexpr int tmem_cols = kG == 3 ? 256 : 128;      // one 64-column S tile per group
    // ring slot k % stages always serves group (k / block) % groups: each group
    // waits on its own slots in order, so a full barrier's parity never aliases
    static_assert(ring_blocks % groups == 0, "ring blocks must be a multiple of the groups");
    static_assert(kA2Block == 4 && groups * 64 <= tmem_cols, "tcgen05 Q K^T: 4-page blocks of 64 keys");
};
constexpr int kA2OStride = 68;                            // floats per row of the O partial
constexpr int kA2MaxSplits = 16;
constexpr int kA2AutoSplits = 8;   // the largest split chosen by default
constexpr int kA2MaxRequests = 65535;   // grid z
constexpr int kA2WsMaxSplits = 256;     // workspace engine: CTAs per (request, KV head)
constexpr int kA2WsSlotFloats = 64 * 64 + 64 + 64 + 64;   // per split: O [64][64], m, l, flag: 17152 bytes

// The split-KV partials of one (request, KV head), S * kA2WsSlotFloats floats:
// the S O partials [64 rows][64] (split order), then the row maxima [64][S]
// and the row sums [64][S] (a row's S values side by side, so one load of a
// warp reads them all), then the S bad-entry flags, then padding.
struct A2WsRegion {
    float *o, *m, *l;
    int *bad;
};
__device__ __forceinline__ A2WsRegion a2_ws_region(float *ws, int r, int nkv, int g, int S)
{
    A2WsRegion w;
    w.o = ws + ((size_t)r * nkv + g) * S * kA2WsSlotFloats;
    w.m = w.o + (size_t)S * 4096;
    w.l = w.m + (size_t)S * 64;
    w.bad = reinterpret_cast<int *>(w.l + (size_t)S * 64);
    return w;
}

struct A2Layout {
    uint32_t q, gate, ring, full, empty, sbar, tslot, o, m, l, flags, total;
};

// groups 1.. leave their O partials over the ring: written only once every
// page has been consumed and every copy has landed
static_assert((A2Shape<3>::groups - 1) * 64 * kA2OStride * 4 <= A2Shape<3>::ring_blocks * kA2Block * kA2PageBytes &&
                  (A2Shape<2>::groups - 1) * 64 * kA2OStride * 4 <= A2Shape<2>::ring_blocks * kA2Block * kA2PageBytes,
              "O partials must fit the ring");

template <int kG>
__host__ __device__ inline A2Layout a2_layout()
{
    using Sh = A2Shape<kG>;
    A2Layout L;
    uint32_t off = 0;
    L.q = off;
    off += 64 * 128;
    L.gate = off;   // the rows' gate heads, bf16 [64 rows][64], loaded with Q
    off += 64 * 128;
    L.ring = off;
    L.o = off;
    off += Sh::ring_blocks * kA2Block * kA2PageBytes;
    L.full = off;
    off += Sh::ring_blocks * 8;
    L.empty = off;
    off += Sh::ring_blocks * 8;
    L.sbar = off;   // per group: its Q K^T (tcgen05) is done
    off += Sh::groups * 8;
    L.tslot = off;  // tensor-memory base address
    off += 8;
    L.m = off;
    off += Sh::groups * 64 * 4;
    L.l = off;
    off += Sh::groups * 64 * 4;
    L.flags = off;
    off += 16;
    L.total = off + 1024;   // alignment slack
    return L;
}

struct Attn2Params {
    const uint16_t *qkv;
    float *ws;               // split-KV partials (workspace engine), else null
    const int32_t *block_table;
    const int32_t *context_lens;
    uint16_t *out;
    int64_t num_pages;
    unsigned long long wait_limit_ns;
    int max_blocks;
    int N;
    int nkv;
    int window;
    int splits;
    float scale_log2;   // softmax scale times log2(e)
    float eps;
};

// One page box of the 5-D cache map (coordinates 0, 0, 0, 0, c4).  `policy`:
// an L2 cache policy (createpolicy); the cache is streamed once, so its lines
// go first and the rest of the working set (q, the partials, the code) stays
// in L2
__device__ __forceinline__ void tma_load_page(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c4,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %3, %3, %3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(0), "r"(c4), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// named barrier 2 over the compute warps only
template <int kG>
__device__ __forceinline__ void a2_compute_bar_sync()
{
    asm volatile("bar.sync 2, %0;" ::"n"(32 * A2Shape<kG>::compute_warps) : "memory");
}

// named barrier 3 over every warp: the ring is drained and free
template <int kG>
__device__ __forceinline__ void a2_ring_done_sync()
{
    asm volatile("bar.sync 3, %0;" ::"n"(A2Shape<kG>::threads) : "memory");
}

// named barrier 4 + grp over the 4 warps of compute group grp
__device__ __forceinline__ void a2_group_bar_sync(int grp)
{
    asm volatile("bar.sync %0, 128;" ::"r"(4 + grp) : "memory");
}

template <int kCols>
__device__ __forceinline__ void a2_tmem_alloc(uint32_t slot_saddr)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
                 "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int kCols>
__device__ __forceinline__ void a2_tmem_dealloc(uint32_t taddr)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kCols)
                 : "memory");
}

// 16 lanes x 64 consecutive 32-bit columns of tensor memory in the layout of
// mma.sync accumulators: register 4 i + e of thread (gq = lane / 4, t = lane % 4)
// holds lane taddr.lane + gq (+ 8 for e >= 2), column taddr.col + 8 i + 2 t + (e & 1).
__device__ __forceinline__ void a2_tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Shared-memory descriptor of a 128-byte-swizzled K-major operand whose
// 8-row groups lie `sbo` bytes apart (a page's K rows of slots 0-7 and 8-15,
// and the next page's, are 2 KB apart in the ring)
__device__ __forceinline__ uint64_t a2_desc_sw128(uint32_t saddr, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address / 16
    d |= (uint64_t)1 << 16;                             // leading offset (unused when swizzled)
    d |= (uint64_t)(sbo >> 4) << 32;                    // stride offset: one 8-row group
    d |= (uint64_t)1 << 46;                             // descriptor version
    d |= (uint64_t)2 << 61;                             // 128-byte swizzle
    return d;
}

// 2^x for x <= 0 (softmax weights): the hardware approximation, subnormal
// results flushed to zero — weights below 2^-126 of the row maximum
__device__ __forceinline__ float a2_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f2bf(float lo, float hi)
{
    return pack_bf16x2(__float2bfloat16_rn(lo), __float2bfloat16_rn(hi));
}

// The gate values at dims 2 lane, 2 lane + 1 of output row `row` of
// (request r, KV head g): gate head 8 g + row % 8 of token row / 8.
__device__ __forceinline__ __nv_bfloat162 a2_gate(const Attn2Params &p, int r, int g, int row, int lane)
{
    const int gate_col = kQPerKv * p.nkv * kHeadDim + 2 * p.nkv * kHeadDim;
    const size_t qrow = (size_t)r * 8 + (row >> 3);
    return *reinterpret_cast<const __nv_bfloat162 *>(p.qkv + qrow * p.N + gate_col +
                                                    (size_t)(8 * g + (row & 7)) * kHeadDim + 2 * lane);
}

// The finish's scalar math on the special-function unit (approximate
// reciprocal, reciprocal square root and exponential, errors ~1e-6 relative,
// far below the BF16 output's 2^-9), in place of the IEEE division and
// square-root sequences: the once-per-CTA tail is shorter (at 32 requests of
// 1K, 30.8 -> 29.0 us a call).
__device__ __forceinline__ float a2_recip(float x) { return x > 0.f ? __fdividef(1.0f, x) : 0.f; }
__device__ __forceinline__ float a2_rnorm(float sum_sq, float eps)
{
    return rsqrtf(sum_sq * (1.0f / kHeadDim) + eps);
}
__device__ __forceinline__ float a2_sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// One output row of (request r, KV head g): o = (o0, o1) at dims 2 lane,
// 2 lane + 1 and its softmax sum lt -> 1/lt, o-norm over the 64 dims (warp
// butterfly), sigmoid gate gt of the row's gate head, bf16 store.
__device__ __forceinline__ void a2_finish_row(const Attn2Params &p, int r, int g, int row, float o0,
                                              float o1, float lt, int lane, __nv_bfloat162 gt)
{
    const int out_cols = kQPerKv * p.nkv * kHeadDim;
    const float inv = a2_recip(lt);
    o0 *= inv;
    o1 *= inv;
    float ss = o0 * o0 + o1 * o1;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rn = a2_rnorm(ss, p.eps);
    const int tok = row >> 3, hj = 8 * g + (row & 7);
    const size_t qrow = (size_t)r * 8 + tok;
    const float s0 = a2_sigmoid(__low2float(gt));
    const float s1 = a2_sigmoid(__high2float(gt));
    reinterpret_cast<uint32_t *>(p.out + qrow * out_cols + (size_t)hj * kHeadDim)[lane] =
        pack_f2bf(o0 * rn * s0, o1 * rn * s1);
}

// The same finish with 8 lanes per row: lane j of the row's group of 8 holds
// dims 8 j .. 8 j + 7 (o = oa | ob, their gate values in gw), so a warp
// finishes 4 rows at once; the o-norm's sum is a 3-level butterfly inside the
// group.  `store` is false for a padding row past the tile.
__device__ __forceinline__ void a2_finish_row8(const Attn2Params &p, int r, int g, int row, float4 oa,
                                               float4 ob, float lt, int j, uint4 gw, bool store)
{
    const int out_cols = kQPerKv * p.nkv * kHeadDim;
    const float inv = a2_recip(lt);
    const float o[8] = {oa.x * inv, oa.y * inv, oa.z * inv, oa.w * inv,
                        ob.x * inv, ob.y * inv, ob.z * inv, ob.w * inv};
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ss += o[k] * o[k];
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rn = a2_rnorm(ss, p.eps);
    const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
    uint32_t res[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float g0 = __uint_as_float(gv[q] << 16), g1 = __uint_as_float(gv[q] & 0xffff0000u);
        const float s0 = a2_sigmoid(g0);
        const float s1 = a2_sigmoid(g1);
        res[q] = pack_f2bf(o[2 * q] * rn * s0, o[2 * q + 1] * rn * s1);
    }
    if (store) {
        const int tok = row >> 3, hj = 8 * g + (row & 7);
        const size_t qrow = (size_t)r * 8 + tok;
        *reinterpret_cast<uint4 *>(p.out + qrow * out_cols + (size_t)hj * kHeadDim + 8 * j) =
            make_uint4(res[0], res[1], res[2], res[3]);
    }
}

// kWorkspace = false: the S CTAs of (request, KV head) form a cluster and merge
// over distributed shared memory.  true: no cluster; each CTA writes its
// partial to its slot of the caller's workspace and attn2_merge_kernel, the
// next grid on the stream, merges the S slots.
template <bool kWorkspace, int kG>
__global__ void __launch_bounds__(A2Shape<kG>::threads, A2Shape<kG>::ctas_per_sm)
    attn2_kernel(const __grid_constant__ CUtensorMap tmKV, const Attn2Params p)
{
    using Sh = A2Shape<kG>;
    constexpr int kGroupsN = Sh::groups, kComputeWarps = Sh::compute_warps, kRing = Sh::ring_blocks;
    extern __shared__ uint8_t a2_smem_dyn[];
    uint8_t *smem = a2_smem_dyn + ((1024u - (smem_u32(a2_smem_dyn) & 1023u)) & 1023u);
    const A2Layout LY = a2_layout<kG>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.splits;
    const uint32_t z = kWorkspace ? blockIdx.x : (S > 1 ? cluster_rank() : 0u);
    const int g = blockIdx.y, r = blockIdx.z;
    const uint32_t sQ = smem_u32(smem + LY.q), sRing = smem_u32(smem + LY.ring);
    const uint32_t full0 = smem_u32(smem + LY.full), empty0 = smem_u32(smem + LY.empty);
    float *o_part = reinterpret_cast<float *>(smem + LY.o);
    float *m_part = reinterpret_cast<float *>(smem + LY.m);
    float *l_part = reinterpret_cast<float *>(smem + LY.l);
    // [0] abort, [1] a table entry of this CTA's pages is outside the cache
    volatile int *s_flags = reinterpret_cast<volatile int *>(smem + LY.flags);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) {   // one full / empty pair per block of pages
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 4);   // the 4 warps of the group that owns the block
        }
        for (int q = 0; q < kGroupsN; ++q) mbar_init(smem_u32(smem + LY.sbar) + 8 * q, 1);
        s_flags[0] = 0;
        s_flags[1] = 0;
        fence_barrier_init();
        griddep_launch_dependents();
    }
    if (warp == 0) a2_tmem_alloc<Sh::tmem_cols>(smem_u32(smem + LY.tslot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();   // q, the cache, the table and the lengths come from earlier kernels

    // ---- the request: length and visible pages ----------------------------
    // Issued together, before anything waits on one of them: the length, the
    // producer's first 32 table entries (without a window they do not depend
    // on the length), and the compute warps' Q and gate tiles.
    const int32_t *bt = p.block_table + (size_t)r * p.max_blocks;
    int first_entry = 0;
    if (warp == kComputeWarps && p.window == 0 && (int)z + lane * S < p.max_blocks) first_entry = bt[z + lane * S];
    const int L = p.context_lens[r];
    if (warp < kComputeWarps) {
        // Q tile [64 rows][64 dims], row 8 i + j = token i, head 8 g + j;
        // 128-byte rows with the chunk XORed by row % 8 (as TMA would); the
        // same rows' gate heads for the finish (no global load at the tail)
        const int gate_col = kQPerKv * p.nkv * kHeadDim + 2 * p.nkv * kHeadDim;
        for (int c = threadIdx.x; c < 512; c += 32 * kComputeWarps) {
            const int row = c >> 3, cc = c & 7;
            const uint16_t *src = p.qkv + ((size_t)r * 8 + (row >> 3)) * p.N + (size_t)(8 * g + (row & 7)) * kHeadDim + 8 * cc;
            const uint4 qv = *reinterpret_cast<const uint4 *>(src);
            const uint4 gv = *reinterpret_cast<const uint4 *>(src + gate_col);
            *reinterpret_cast<uint4 *>(smem + LY.q + row * 128 + ((cc ^ (row & 7)) << 4)) = qv;
            *reinterpret_cast<uint4 *>(smem + LY.gate + row * 128 + 16 * cc) = gv;
        }
        // the tensor cores read Q through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    const int nblk = (L + kPageSlots - 1) / kPageSlots;
    const bool len_ok = L >= 8 && nblk <= p.max_blocks;
    if (!len_ok && threadIdx.x == 0 && z == 0 && g == 0) atomicOr(&g_status, QKVF_STATUS_BAD_REQUEST);
    const int p_first = (p.window > 0 && L - 8 - p.window + 1 > 0) ? (L - 8 - p.window + 1) / kPageSlots : 0;
    const int p_last = len_ok ? (L - 1) / kPageSlots : -1;
    const bool req_ok = len_ok;
    const int first_mine = p_first + (int)z;
    const int npages = (len_ok && first_mine <= p_last) ? (p_last - first_mine) / S + 1 : 0;

    if (warp == kComputeWarps) {
        // ---- produce: K and V boxes of this CTA's pages -------------------
        // The table entries come in 32 at a time (lane l holds page c + l of
        // chunk c), one chunk ahead of the copies, so no copy waits on a
        // table read.  Per block of 4 pages: lane 0 waits for the ring block
        // and arms its full barrier with the block's bytes, then the lanes
        // holding the block's pages issue their copies side by side, one
        // 4-KB box per page.  An
        // entry outside the cache is flagged (the request's rows are then
        // skipped by every rank) and page 0 copied instead, so the ring's
        // accounting does not change.
        if (lane == 0) tma_prefetch_map(&tmKV);
        const uint64_t pol_kv = policy_evict_first();   // the cache is streamed once
        int issued = 0;   // blocks
        unsigned bad = 0u;
        bool stop = false;
        // (with a window the first entries wait for the length)
        int next = lane < npages ? (p.window == 0 ? first_entry : bt[first_mine + lane * S]) : 0;
        for (int c = 0; c < npages && !stop; c += 32) {
            int page = next;
            if (c + 32 + lane < npages) next = bt[first_mine + (c + 32 + lane) * S];
            if (c + lane < npages && (page < 0 || page >= p.num_pages)) {
                bad = 1u;
                page = 0;
            }
            const int c_end = npages - c < 32 ? npages : c + 32;
            for (int k0 = c; k0 < c_end; k0 += kA2Block) {
                const int jb = k0 / kA2Block, rb = jb % kRing, use = jb / kRing;
                const int nb = npages - k0 < kA2Block ? npages - k0 : kA2Block;
                int ok = 1;
                if (lane == 0) {
                    ok = use == 0 || bounded_wait(empty0 + 8 * rb, (uint32_t)((use - 1) & 1),
                                                  s_flags, p.wait_limit_ns, true);
                    if (ok) mbar_expect_tx(full0 + 8 * rb, (uint32_t)nb * kA2PageBytes);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    stop = true;
                    break;
                }
                const int b = c + lane - k0;   // this lane's page within the block
                if (b >= 0 && b < nb) {   // page b of the block
                    const uint32_t blk = sRing + (uint32_t)rb * (kA2Block * kA2PageBytes);
                    tma_load_page(blk + (uint32_t)b * kA2PageBytes, &tmKV, full0 + 8 * rb, page * p.nkv + g, pol_kv);
                }
                ++issued;
            }
        }
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0) {
            if (bad) {
                s_flags[1] = 1;
                atomicOr(&g_status, QKVF_STATUS_BAD_REQUEST);
            }
            if (s_flags[0]) {   // drain our copies before the ring is reused or we leave
                const int first = issued > kRing ? issued - kRing : 0;
                for (int j = first; j < issued; ++j)
                    bounded_wait(full0 + 8 * (j % kRing), (uint32_t)((j / kRing) & 1),
                                 s_flags, p.wait_limit_ns, false);
            }
        }
        __syncwarp();
        a2_ring_done_sync<kG>();
    } else {
        // ---- compute: group grp = warp / 4 takes blocks grp, grp + G, ... ----
        const int tid = threadIdx.x;
        const int grp = warp >> 2, wig = warp & 3;   // group, warp in group (rows 16 wig ..)
        a2_compute_bar_sync<kG>();   // the Q tile is in shared memory
        const int gq = lane >> 2, t = lane & 3;
        // tcgen05 Q K^T: the group's S tile [64 rows x 64 keys] in tensor memory
        // columns 64 grp.., rows 16 w .. 16 w + 15 in lanes 32 w .. 32 w + 15;
        // column 16 b + s is slot s of the block's page b
        const uint32_t sbar = smem_u32(smem + LY.sbar) + 8 * grp;
        const uint32_t tS = *reinterpret_cast<volatile uint32_t *>(smem + LY.tslot) + 64u * grp;
        const bool issuer = wig == 0 && lane == 0;
        uint32_t sph = 0;            // phase of sbar this block waits for
        int committed = 0, observed = 0;   // the issuer's commits, and those it saw complete

        // this thread's rows: 16 wig + gq (token 2 wig) and 16 wig + gq + 8 (token 2 wig + 1)
        const int pos_a = L - 8 + 2 * wig, pos_b = pos_a + 1;
        const int lo_a = p.window > 0 ? pos_a - p.window + 1 : 0;
        const int lo_b = p.window > 0 ? pos_b - p.window + 1 : 0;
        // keys every row sees: [edge_lo, edge_hi]; a page inside needs no mask
        const int edge_lo = p.window > 0 ? L - p.window : 0, edge_hi = L - 8;
        float o[8][4];
#pragma unroll
        for (int nd = 0; nd < 8; ++nd)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

        // V: this lane's ldmatrix.trans row, slot (lane & 7) + 8 ((lane >> 3) & 1) of a page
        const uint32_t v_row = (uint32_t)((lane & 7) * 128 + ((lane >> 3) & 1) * 2048);
        const uint32_t v_hi = (uint32_t)(lane >> 4);
        const uint32_t sw = (uint32_t)(lane & 7);

        // blocks of up to kA2Block pages (16 kA2Block keys): one softmax
        // reduction and one rescale of O per block, independent mma chains
        for (int k0 = grp * kA2Block; k0 < npages; k0 += kGroupsN * kA2Block) {
            const int nb = npages - k0 < kA2Block ? npages - k0 : kA2Block;   // same for every lane
            const int jb = k0 / kA2Block, rb = jb % kRing;
            const uint32_t ph = (uint32_t)((jb / kRing) & 1);
            // the block's keys rise with its pages: the first and the last key
            // decide whether every row sees all of them
            const int key_first = (first_mine + k0 * S) * kPageSlots;
            const int key_last = (first_mine + (k0 + nb - 1) * S) * kPageSlots + kPageSlots - 1;
            const bool inside = nb == kA2Block && key_first >= edge_lo && key_last <= edge_hi;
            bool landed = mbar_try_wait(full0 + 8 * rb, ph) ||
                          bounded_wait(full0 + 8 * rb, ph, s_flags, p.wait_limit_ns, true);
            // the block's 4 pages; the 8-row groups of K (and of V) 2 KB apart
            const uint32_t kreg = sRing + (uint32_t)rb * (kA2Block * kA2PageBytes);
            // every warp of the group is past the previous block's tcgen05.ld
            tc_fence_before();
            a2_group_bar_sync(grp);
            if (issuer && landed) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // K = 16 dims per instruction: 32 bytes along the rows
                    umma_bf16(tS, umma_desc_sw128(sQ + 32u * kk), a2_desc_sw128(kreg + 32u * kk, 2048),
                              umma_idesc_bf16(64, 64), kk != 0 ? 1u : 0u);
                umma_commit(sbar);
                ++committed;
            }
            const bool s_ok = mbar_try_wait(sbar, sph) || bounded_wait(sbar, sph, s_flags, p.wait_limit_ns, true);
            sph ^= 1u;
            if (issuer && s_ok) observed = committed;
            landed = landed && s_ok;
            if (__all_sync(0xffffffffu, landed)) {
                float sc[2 * kA2Block][4];
                tc_fence_after();
                uint32_t rr[32];
                a2_tmem_ld_16x256b_x8(tS + ((uint32_t)(32 * wig) << 16), rr);
                tmem_ld_wait();
#pragma unroll
                for (int nt = 0; nt < 2 * kA2Block; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] = __uint_as_float(rr[4 * nt + e]);
                // (near the edges) mask: element e of tile nt = 2 b + h is key
                // key0(b) + 8 h + 2 t + (e & 1), row a for e < 2
                if (!inside) {
#pragma unroll
                    for (int b = 0; b < kA2Block; ++b) {
                        const int key0 = (first_mine + (k0 + b) * S) * kPageSlots;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int key = key0 + 8 * h + 2 * t + (e & 1);
                                const bool ok = b < nb && (e >= 2 ? (key >= lo_b && key <= pos_b)
                                                                  : (key >= lo_a && key <= pos_a));
                                if (!ok) sc[2 * b + h][e] = -INFINITY;
                            }
                    }
                }
                // block maxima of the raw scores (the scale is positive), as trees
                float tm[2 * kA2Block][2];
#pragma unroll
                for (int nt = 0; nt < 2 * kA2Block; ++nt) {
                    tm[nt][0] = fmaxf(sc[nt][0], sc[nt][1]);
                    tm[nt][1] = fmaxf(sc[nt][2], sc[nt][3]);
                }
#pragma unroll
                for (int w = kA2Block; w >= 1; w >>= 1)
#pragma unroll
                    for (int nt = 0; nt < w; ++nt) {
                        tm[nt][0] = fmaxf(tm[nt][0], tm[nt + w][0]);
                        tm[nt][1] = fmaxf(tm[nt][1], tm[nt + w][1]);
                    }
                float mx_a = tm[0][0] * p.scale_log2, mx_b = tm[0][1] * p.scale_log2;
#pragma unroll
                for (int off = 1; off <= 2; off <<= 1) {
                    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
                    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
                }
                const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
                const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
                const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
                // O and the sums are rescaled only when some row's maximum grew
                // (otherwise the factor is exactly 1 and the product the same)
                const bool grew = __any_sync(0xffffffffu, mn_a != m_a || mn_b != m_b);
                // weights 2^(scale s - base), one FMA and one ex2 each; sums as trees
                float ts[2 * kA2Block][2];
#pragma unroll
                for (int nt = 0; nt < 2 * kA2Block; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sc[nt][e] = a2_ex2(fmaf(sc[nt][e], p.scale_log2, e >= 2 ? -base_b : -base_a));
                    ts[nt][0] = sc[nt][0] + sc[nt][1];
                    ts[nt][1] = sc[nt][2] + sc[nt][3];
                }
#pragma unroll
                for (int w = kA2Block; w >= 1; w >>= 1)
#pragma unroll
                    for (int nt = 0; nt < w; ++nt) {
                        ts[nt][0] += ts[nt + w][0];
                        ts[nt][1] += ts[nt + w][1];
                    }
                if (grew) {
                    const float al_a = a2_ex2(m_a - base_a), al_b = a2_ex2(m_b - base_b);
                    l_a = l_a * al_a;
                    l_b = l_b * al_b;
#pragma unroll
                    for (int nd = 0; nd < 8; ++nd) {
                        o[nd][0] *= al_a;
                        o[nd][1] *= al_a;
                        o[nd][2] *= al_b;
                        o[nd][3] *= al_b;
                    }
                }
                l_a = l_a + ts[0][0];
                l_b = l_b + ts[0][1];
                m_a = mn_a;
                m_b = mn_b;
#pragma unroll
                for (int b = 0; b < kA2Block; ++b) {
                    if (b < nb) {
                        const uint32_t vbox = kreg + (uint32_t)b * kA2PageBytes + 1024;   // page b's V rows 0-7
                        // P (rows a / b x the page's 16 keys) as the A fragment of PV
                        const uint32_t pa0 = pack_f2bf(sc[2 * b][0], sc[2 * b][1]);
                        const uint32_t pa1 = pack_f2bf(sc[2 * b][2], sc[2 * b][3]);
                        const uint32_t pa2 = pack_f2bf(sc[2 * b + 1][0], sc[2 * b + 1][1]);
                        const uint32_t pa3 = pack_f2bf(sc[2 * b + 1][2], sc[2 * b + 1][3]);
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {   // dims 16 q2 .. 16 q2 + 15
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_trans(vbox + v_row + ((((uint32_t)(2 * q2) + v_hi) ^ sw) << 4), b0, b1, b2, b3);
                            mma_bf16_16816(o[2 * q2], pa0, pa1, pa2, pa3, b0, b1);
                            mma_bf16_16816(o[2 * q2 + 1], pa0, pa1, pa2, pa3, b2, b3);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * rb);
        }
        if (issuer && committed != observed)   // an abandoned wait: let the MMAs finish first
            bounded_wait(sbar, (uint32_t)((committed - 1) & 1), s_flags, p.wait_limit_ns, false);
        tc_fence_before();
        a2_ring_done_sync<kG>();   // every group is past the ring; the producer has drained
        tc_fence_after();
        if (warp == 0) a2_tmem_dealloc<Sh::tmem_cols>(*reinterpret_cast<volatile uint32_t *>(smem + LY.tslot));
        // whole-row sums across the four threads of a row
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
        }
        // Fold the groups' partials into group 0's registers, in group order:
        // groups 1.. leave theirs in shared memory (over the drained ring)
        const int ra = wig * 16 + gq, rb = ra + 8;
        if (grp > 0) {
            float *og = o_part + grp * (64 * kA2OStride);
#pragma unroll
            for (int nd = 0; nd < 8; ++nd) {
                *reinterpret_cast<float2 *>(og + ra * kA2OStride + 8 * nd + 2 * t) = make_float2(o[nd][0], o[nd][1]);
                *reinterpret_cast<float2 *>(og + rb * kA2OStride + 8 * nd + 2 * t) = make_float2(o[nd][2], o[nd][3]);
            }
            if (t == 0) {
                m_part[grp * 64 + ra] = m_a;
                m_part[grp * 64 + rb] = m_b;
                l_part[grp * 64 + ra] = l_a;
                l_part[grp * 64 + rb] = l_b;
            }
        }
        a2_compute_bar_sync<kG>();
        if (grp == 0) {
            float w_a[kGroupsN], w_b[kGroupsN];
            {
                float mg_a[kGroupsN], mg_b[kGroupsN];
                mg_a[0] = m_a;
                mg_b[0] = m_b;
#pragma unroll
                for (int gg = 1; gg < kGroupsN; ++gg) {
                    mg_a[gg] = m_part[gg * 64 + ra];
                    mg_b[gg] = m_part[gg * 64 + rb];
                }
                float M_a = -INFINITY, M_b = -INFINITY;
#pragma unroll
                for (int gg = 0; gg < kGroupsN; ++gg) {
                    M_a = fmaxf(M_a, mg_a[gg]);
                    M_b = fmaxf(M_b, mg_b[gg]);
                }
                const float base_a = M_a == -INFINITY ? 0.f : M_a, base_b = M_b == -INFINITY ? 0.f : M_b;
#pragma unroll
                for (int gg = 0; gg < kGroupsN; ++gg) {
                    w_a[gg] = exp2f(mg_a[gg] - base_a);
                    w_b[gg] = exp2f(mg_b[gg] - base_b);
                }
                m_a = M_a;
                m_b = M_b;
            }
            float lt_a = 0.f, lt_b = 0.f;
            lt_a = lt_a + l_a * w_a[0];
            lt_b = lt_b + l_b * w_b[0];
#pragma unroll
            for (int gg = 1; gg < kGroupsN; ++gg) {
                lt_a = lt_a + l_part[gg * 64 + ra] * w_a[gg];
                lt_b = lt_b + l_part[gg * 64 + rb] * w_b[gg];
            }
            l_a = lt_a;
            l_b = lt_b;
#pragma unroll
            for (int nd = 0; nd < 8; ++nd) {
                float f0 = 0.f, f1 = 0.f, f2 = 0.f, f3 = 0.f;
                f0 = f0 + o[nd][0] * w_a[0];
                f1 = f1 + o[nd][1] * w_a[0];
                f2 = f2 + o[nd][2] * w_b[0];
                f3 = f3 + o[nd][3] * w_b[0];
#pragma unroll
                for (int gg = 1; gg < kGroupsN; ++gg) {
                    const float *og = o_part + gg * (64 * kA2OStride);
                    const float2 va = *reinterpret_cast<const float2 *>(og + ra * kA2OStride + 8 * nd + 2 * t);
                    const float2 vb = *reinterpret_cast<const float2 *>(og + rb * kA2OStride + 8 * nd + 2 * t);
                    f0 = f0 + va.x * w_a[gg];
                    f1 = f1 + va.y * w_a[gg];
                    f2 = f2 + vb.x * w_b[gg];
                    f3 = f3 + vb.y * w_b[gg];
                }
                o[nd][0] = f0;
                o[nd][1] = f1;
                o[nd][2] = f2;
                o[nd][3] = f3;
            }
            if constexpr (kWorkspace) {
                // ---- publish this CTA's partial: O [64][64], m, l, the bad-entry flag ----
                const A2WsRegion wr = a2_ws_region(p.ws, r, p.nkv, g, S);
                float *slot = wr.o + (size_t)z * 4096;
#pragma unroll
                for (int nd = 0; nd < 8; ++nd) {
                    __stcg(reinterpret_cast<float2 *>(slot + ra * 64 + 8 * nd + 2 * t), make_float2(o[nd][0], o[nd][1]));
                    __stcg(reinterpret_cast<float2 *>(slot + rb * 64 + 8 * nd + 2 * t), make_float2(o[nd][2], o[nd][3]));
                }
                if (t == 0) {
                    __stcg(wr.m + ra * S + z, m_a);
                    __stcg(wr.m + rb * S + z, m_b);
                    __stcg(wr.l + ra * S + z, l_a);
                    __stcg(wr.l + rb * S + z, l_b);
                }
                if (tid == 0) __stcg(wr.bad + z, s_flags[1]);
            } else {
                // the CTA's partial for the ranks' merge or the finish: slice 0
#pragma unroll
                for (int nd = 0; nd < 8; ++nd) {
                    *reinterpret_cast<float2 *>(o_part + ra * kA2OStride + 8 * nd + 2 * t) = make_float2(o[nd][0], o[nd][1]);
                    *reinterpret_cast<float2 *>(o_part + rb * kA2OStride + 8 * nd + 2 * t) = make_float2(o[nd][2], o[nd][3]);
                }
                if (t == 0) {
                    m_part[ra] = m_a;
                    m_part[rb] = m_b;
                    l_part[ra] = l_a;
                    l_part[rb] = l_b;
                }
            }
        }
    }
    __syncthreads();
    if constexpr (!kWorkspace) {
        if (S > 1) cluster_sync_all();

        // a request with an entry outside the cache on any rank is skipped by all
        bool table_ok = true;
        if (req_ok) {
            unsigned bad_rank = 0u;
            if (S > 1) {
                if (lane < S) bad_rank = ld_cluster_u32(map_to_rank(smem_u32(smem + LY.flags) + 4u, (uint32_t)lane));
            } else if (lane == 0) {
                bad_rank = (unsigned)s_flags[1];
            }
            table_ok = !__any_sync(0xffffffffu, bad_rank != 0u);
        }

        // ---- merge the ranks' partials, o-norm, gate, store (64 / S rows each) ----
        if (req_ok && table_ok && S == 1) {
            // one CTA holds the whole partial: 8 lanes per row, 4 rows per warp at a time
            const int sub = lane >> 3, j = lane & 7;
            for (int base = 4 * warp; base < 64; base += 4 * (kComputeWarps + 1)) {
                const int row = base + sub;
                const int rr = row < 64 ? row : 63;
                const float4 oa = *reinterpret_cast<const float4 *>(o_part + rr * kA2OStride + 8 * j);
                const float4 ob = *reinterpret_cast<const float4 *>(o_part + rr * kA2OStride + 8 * j + 4);
                const uint4 gw = *reinterpret_cast<const uint4 *>(smem + LY.gate + rr * 128 + 16 * j);
                a2_finish_row8(p, r, g, row, oa, ob, l_part[rr], j, gw, row < 64);
            }
        } else if (req_ok && table_ok) {
            const int rows = 64 / S;
            const uint32_t o_addr = smem_u32(o_part), m_addr = smem_u32(m_part), l_addr = smem_u32(l_part);
            for (int i = warp; i < rows; i += kComputeWarps + 1) {
                const int row = (int)z * rows + i;
                const __nv_bfloat162 gt = *reinterpret_cast<const __nv_bfloat162 *>(smem + LY.gate + row * 128 + 4 * lane);
                // the ranks' partials in rank order (short loops: a fully unrolled
                // merge over every possible rank cost ~3000 cycles a row)
                float lt, o0, o1;
                {
                    float M = -INFINITY;
#pragma unroll 4
                    for (int src = 0; src < S; ++src)
                        M = fmaxf(M, ld_cluster_f32(map_to_rank(m_addr + 4u * row, (uint32_t)src)));
                    const float base = M == -INFINITY ? 0.f : M;
                    lt = 0.f;
                    o0 = 0.f;
                    o1 = 0.f;
#pragma unroll 4
                    for (int src = 0; src < S; ++src) {
                        const float w = exp2f(ld_cluster_f32(map_to_rank(m_addr + 4u * row, (uint32_t)src)) - base);
                        const float lk = ld_cluster_f32(map_to_rank(l_addr + 4u * row, (uint32_t)src));
                        const float2 ov =
                            ld_cluster_f2(map_to_rank(o_addr + 4u * (row * kA2OStride + 2 * lane), (uint32_t)src));
                        lt = lt + lk * w;
                        o0 = o0 + ov.x * w;
                        o1 = o1 + ov.y * w;
                    }
                }
                a2_finish_row(p, r, g, row, o0, o1, lt, lane, gt);
            }
        }
        if (S > 1) cluster_sync_all();   // no CTA leaves while its partials may still be read
    }
}

// Merge of the split-KV engine, the grid after attn2_kernel<true> on the
// stream: one warp per output row of (request, KV head).  Lane l holds the
// maximum and sum of split l (of l, l + 32, ... past 32 splits); the row's
// maximum and sum are warp reductions in a fixed order; O is summed over the
// splits in split order, 32 splits' loads in flight per batch; then o-norm,
// gate, store.  Every load of the first batch is issued before any is used
// (one round trip); a row's maxima, sums and flags are one coalesced load
// each (scattered per-split loads doubled the round trip at 19 splits).
constexpr int kA2MergeWarps = 4;

__global__ void __launch_bounds__(32 * kA2MergeWarps) attn2_merge_kernel(const Attn2Params p)
{
    __shared__ float w_sh[kA2MergeWarps][kA2WsMaxSplits];
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();   // the partials (and, transitively, q and the gate) are written
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kA2MergeWarps + warp, g = blockIdx.y, r = blockIdx.z;
    const int S = p.splits;
    const A2WsRegion wr = a2_ws_region(p.ws, r, p.nkv, g, S);
    const float *mrow = wr.m + row * S, *lrow = wr.l + row * S;
    const int L = p.context_lens[r];
    const __nv_bfloat162 gt = a2_gate(p, r, g, row, lane);
    float m0 = -INFINITY, l0 = 0.f;
    unsigned bad = 0u;
    if (lane < S) {
        m0 = __ldcg(mrow + lane);
        l0 = __ldcg(lrow + lane);
        bad = (unsigned)__ldcg(wr.bad + lane);
    }
    float2 v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j < S) v[j] = __ldcg(reinterpret_cast<const float2 *>(wr.o + (size_t)j * 4096 + row * 64 + 2 * lane));
    float M = m0;
    for (int src = lane + 32; src < S; src += 32) M = fmaxf(M, __ldcg(mrow + src));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float base = M == -INFINITY ? 0.f : M;
    float lt = 0.f;
    if (lane < S) {
        const float w = exp2f(m0 - base);
        w_sh[warp][lane] = w;
        lt = lt + l0 * w;
    }
    for (int src = lane + 32; src < S; src += 32) {
        const float w = exp2f(__ldcg(mrow + src) - base);
        w_sh[warp][src] = w;
        lt = lt + __ldcg(lrow + src) * w;
        bad |= (unsigned)__ldcg(wr.bad + src);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    __syncwarp();
    float o0 = 0.f, o1 = 0.f;
    for (int s0 = 0; s0 < S; s0 += 32) {
        if (s0 > 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (s0 + j < S)
                    v[j] = __ldcg(reinterpret_cast<const float2 *>(wr.o + (size_t)(s0 + j) * 4096 + row * 64 + 2 * lane));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (s0 + j < S) {
                const float w = w_sh[warp][s0 + j];
                o0 = o0 + v[j].x * w;
                o1 = o1 + v[j].y * w;
            }
        }
    }
    // a bad request, or a page outside the cache on any split: rows skipped
    const bool req_ok = L >= 8 && (L + kPageSlots - 1) / kPageSlots <= p.max_blocks;
    if (req_ok && !__any_sync(0xffffffffu, bad != 0u)) a2_finish_row(p, r, g, row, o0, o1, lt, lane, gt);
}

int encode_kv_map(const uint16_t *kv_cache, int64_t num_pages, int nkv, CUtensorMap *m)
{
    // the cache [pages * nkv][2][8 slots][2 halves][64] seen as dim 0 = 64
    // elements of a half, dim 1 = slot % 8 (256 B apart), dim 2 = K / V half
    // (128 B apart), dim 3 = slot / 8 (2 KB apart), dim 4 = (page, KV head).
    // A {64, 8, 2, 2, 1} box is one page of one KV head in shared memory as
    // K of slots 0-7, V of slots 0-7, K of slots 8-15, V of slots 8-15, 128
    // bytes a row, swizzled
    const cuuint64_t dims[5] = {64, 8, 2, 2, (cuuint64_t)num_pages * nkv};
    const cuuint64_t strides[4] = {256, 128, 2048, (cuuint64_t)kPageSlots * kSlotWidth * 2};
    const cuuint32_t box[5] = {64, 8, 2, 2, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, (void *)kv_cache, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? QKVF_OK
               : QKVF_ERR_CUDA;
}

const char *check_attn2_args(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                             const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                             int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                             uint16_t *out, int *code)
{
    *code = QKVF_ERR_TOKENS;
    if (num_reqs < 0 || num_reqs > kA2MaxRequests) return "num_reqs must be 0..65535";
    *code = QKVF_ERR_SHAPE;
    if (num_kv_heads < 1 || num_kv_heads > 64) return "num_kv_heads must be 1..64";
    if (N != 2 * (kQPerKv + 1) * kHeadDim * num_kv_heads)
        return "N must be 1152 * num_kv_heads: rows [q | k | v | gate]";
    *code = QKVF_ERR_SIZES;
    if (num_pages < 1 || num_pages * num_kv_heads > (int64_t(1) << 31)) return "num_pages * num_kv_heads must be 1..2^31";
    if (max_blocks < 1 || max_blocks > (1 << 24)) return "max_blocks must be 1..2^24";
    *code = QKVF_ERR_ARG;
    if (window < 0) return "window must be >= 0 (0: none)";
    if (!(scale > 0.f) || !(eps > 0.f) || eps > 1.f) return "scale must be > 0 and eps in (0, 1]";
    *code = QKVF_OK;
    if (num_reqs == 0) return nullptr;
    *code = QKVF_ERR_NULL;
    if (!qkv || !kv_cache || !block_table || !context_lens || !out) return "a required pointer is NULL";
    *code = QKVF_ERR_ALIGN;
    if (!aligned(qkv, 16) || !aligned(kv_cache, 16) || !aligned(out, 16))
        return "qkv, kv_cache and out must be 16-byte aligned";
    if (!aligned(block_table, 4) || !aligned(context_lens, 4)) return "block_table and context_lens must be int32-aligned";
    *code = QKVF_ERR_ARG;
    const size_t out_b = (size_t)num_reqs * 8 * kQPerKv * num_kv_heads * kHeadDim * 2;
    const size_t qkv_b = (size_t)num_reqs * 8 * N * 2;
    const size_t cache_b = (size_t)num_pages * num_kv_heads * kPageSlots * kSlotWidth * 2;
    const void *ins[] = {qkv, kv_cache, block_table, context_lens};
    const size_t in_b[] = {qkv_b, cache_b, (size_t)num_reqs * max_blocks * 4, (size_t)num_reqs * 4};
    for (int i = 0; i < 4; ++i)
        if (overlap(ins[i], in_b[i], out, out_b)) return "an input overlaps out";
    *code = QKVF_OK;
    return nullptr;
}

// CTAs per (request, KV head): doubled while the grid stays within one CTA
// per SM and every split keeps at least two pages, up to clusters of 8 (with
// a CTA filling an SM's shared memory, fewer clusters of 16 than GPCs fit at
// once).  The pages a request can need are its table's width, or with a
// window W the at most W + 7 keys some row sees, over at most
// ceil((W + 7) / 16) + 1 pages.
int attn2_splits_for(int num_reqs, int nkv, int max_blocks, int window, int sms)
{
    int64_t pages = max_blocks;
    if (window > 0) {
        const int64_t wp = ((int64_t)window + 7 + kPageSlots - 1) / kPageSlots + 1;
        if (wp < pages) pages = wp;
    }
    int s = 1;
    while (s < kA2AutoSplits && (int64_t)num_reqs * nkv * s * 2 <= sms && pages >= 4 * (int64_t)s) s *= 2;
    return s;
}

// Split-KV engine: CTAs per (request, KV head) so that the grid covers the
// SMs once (R * nkv * S <= SM count), each keeping two or more of the pages a
// row can see.
int attn2_split_kv_splits_for(int num_reqs, int nkv, int max_blocks, int window, int sms)
{
    int64_t pages = max_blocks;
    if (window > 0) {
        const int64_t wp = ((int64_t)window + 7 + kPageSlots - 1) / kPageSlots + 1;
        if (wp < pages) pages = wp;
    }
    int64_t s = sms / ((int64_t)num_reqs * nkv);
    if (s > pages / 2) s = pages / 2;
    if (s > kA2WsMaxSplits) s = kA2WsMaxSplits;
    return s < 1 ? 1 : (int)s;
}

// Workspace of the split-KV engine: R * nkv * S partials of 17152 bytes
// (O [64][64], the 64 row maxima and sums, the bad-entry flag; FP32), laid
// out per (request, KV head) as a2_ws_region describes.
size_t a2_workspace_bytes(int num_reqs, int nkv, int splits)
{
    return (size_t)num_reqs * nkv * splits * kA2WsSlotFloats * 4;
}

bool prepare_attn2_kernel()
{
    const int smem = (int)a2_layout<3>().total;
    return cudaFuncSetAttribute((const void *)attn2_kernel<false, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem) == cudaSuccess &&
           cudaFuncSetAttribute((const void *)attn2_kernel<false, 3>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
           cudaFuncSetAttribute((const void *)attn2_kernel<true, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem) == cudaSuccess &&
           cudaFuncSetAttribute((const void *)attn2_kernel<false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)a2_layout<2>().total) == cudaSuccess;
}

// workspace == null: the cluster engine (splits 1..16, a power of two);
// otherwise the split-KV engine over that workspace (splits 1..256).  A
// direct launch (one split, no workspace) with more (request, KV head) pairs
// than SMs takes the two-CTA-per-SM shape, so all of its CTAs run in one wave.
int launch_attn2(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                 const int32_t *block_table, int max_blocks, const int32_t *context_lens, int num_reqs,
                 int N, int num_kv_heads, int window, float scale, float eps, uint16_t *out, int splits,
                 void *workspace, int sms, void *stream)
{
    CUtensorMap m;
    int rc = encode_kv_map(kv_cache, num_pages, num_kv_heads, &m);
    if (rc != QKVF_OK) return rc;
    const bool ws = workspace != nullptr;
    Attn2Params prm;
    prm.qkv = qkv;
    prm.ws = static_cast<float *>(workspace);
    prm.block_table = block_table;
    prm.context_lens = context_lens;
    prm.out = out;
    prm.num_pages = num_pages;
    prm.wait_limit_ns = g_wait_limit_ns;
    prm.max_blocks = max_blocks;
    prm.N = N;
    prm.nkv = num_kv_heads;
    prm.window = window;
    prm.splits = splits;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.eps = eps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)splits, (unsigned)num_kv_heads, (unsigned)num_reqs);
    const bool two_per_sm = !ws && splits == 1 && (int64_t)num_reqs * num_kv_heads > sms;
    cfg.blockDim = dim3(two_per_sm ? A2Shape<2>::threads : A2Shape<3>::threads, 1, 1);
    cfg.dynamicSmemBytes = two_per_sm ? a2_layout<2>().total : a2_layout<3>().total;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (!ws && splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)splits;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    cudaError_t e = ws ? cudaLaunchKernelEx(&cfg, attn2_kernel<true, 3>, m, prm)
                       : two_per_sm ? cudaLaunchKernelEx(&cfg, attn2_kernel<false, 2>, m, prm)
                                    : cudaLaunchKernelEx(&cfg, attn2_kernel<false, 3>, m, prm);
    if (e == cudaSuccess && ws) {   // the merge, behind the partials
        cudaLaunchConfig_t mc = {};
        mc.gridDim = dim3(64 / kA2MergeWarps, (unsigned)num_kv_heads, (unsigned)num_reqs);
        mc.blockDim = dim3(32 * kA2MergeWarps, 1, 1);
        mc.stream = (cudaStream_t)stream;
        // PDL lets the merge's CTAs start on SMs the page grid leaves idle;
        // when it covers every SM they cannot start before its CTAs exit, and
        // the plain stream order releases the merge sooner (one 32K request,
        // 19 splits on 152 SMs: 20.6 -> 20.1 us a call)
        const bool idle_sms = (int64_t)num_reqs * num_kv_heads * splits < sms;
        cudaLaunchAttribute ma;
        ma.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        ma.val.programmaticStreamSerializationAllowed = g_pdl && idle_sms ? 1 : 0;
        mc.attrs = &ma;
        mc.numAttrs = 1;
        e = cudaLaunchKernelEx(&mc, attn2_merge_kernel, prm);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QKVF_ERR_CUDA;
    }
    return QKVF_OK;
}

}  // namespace qkvf

extern "C" {

int attn2(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
          const int32_t *block_table, int max_blocks, const int32_t *context_lens, int num_reqs,
          int N, int num_kv_heads, int window, float scale, float eps, uint16_t *out, void *stream)
{
    int code;
    if (qkvf::check_attn2_args(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                               num_reqs, N, num_kv_heads, window, scale, eps, out, &code))
        return code;
    if (num_reqs == 0) return QKVF_OK;
    qkvf::DeviceState *d;
    const int rc = qkvf::probe_device(&d);
    if (rc != QKVF_OK) return rc;
    const int splits = qkvf::attn2_splits_for(num_reqs, num_kv_heads, max_blocks, window, d->sms);
    return qkvf::launch_attn2(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                              num_reqs, N, num_kv_heads, window, scale, eps, out, splits, nullptr, d->sms, stream);
}

const char *attn2_unsupported(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                              const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                              int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                              uint16_t *out)
{
    int code;
    const char *why = qkvf::check_attn2_args(qkv, kv_cache, num_pages, block_table, max_blocks,
                                             context_lens, num_reqs, N, num_kv_heads, window, scale,
                                             eps, out, &code);
    if (why) return why;
    qkvf::DeviceState *d;
    const int rc = qkvf::probe_device(&d);
    return rc == QKVF_OK ? nullptr : qkv_front_strerror(rc);
}

int attn2_launch_splits(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                        const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                        int num_reqs, int N, int num_kv_heads, int window, float scale, float eps,
                        uint16_t *out, int splits, void *stream)
{
    int code;
    if (qkvf::check_attn2_args(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                               num_reqs, N, num_kv_heads, window, scale, eps, out, &code))
        return code;
    if (splits != 1 && splits != 2 && splits != 4 && splits != 8 && splits != 16) return QKVF_ERR_VARIANT;
    if (num_reqs == 0) return QKVF_OK;
    qkvf::DeviceState *d;
    const int rc = qkvf::probe_device(&d);
    if (rc != QKVF_OK) return rc;
    return qkvf::launch_attn2(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                              num_reqs, N, num_kv_heads, window, scale, eps, out, splits, nullptr, d->sms, stream);
}

int attn2_splits(int num_reqs, int num_kv_heads, int max_blocks, int window)
{
    if (num_reqs < 1 || num_kv_heads < 1 || max_blocks < 1 || window < 0) return 0;
    qkvf::DeviceState *d;
    if (qkvf::probe_device(&d) != QKVF_OK) return 0;
    return qkvf::attn2_splits_for(num_reqs, num_kv_heads, max_blocks, window, d->sms);
}

size_t attn2_split_kv_workspace_bytes(int num_reqs, int num_kv_heads, int splits)
{
    if (num_reqs < 1 || num_reqs > qkvf::kA2MaxRequests || num_kv_heads < 1 || num_kv_heads > 64 ||
        splits < 1 || splits > qkvf::kA2WsMaxSplits)
        return 0;
    return qkvf::a2_workspace_bytes(num_reqs, num_kv_heads, splits);
}

int attn2_split_kv_splits(int num_reqs, int num_kv_heads, int max_blocks, int window)
{
    if (num_reqs < 1 || num_kv_heads < 1 || max_blocks < 1 || window < 0) return 0;
    qkvf::DeviceState *d;
    if (qkvf::probe_device(&d) != QKVF_OK) return 0;
    return qkvf::attn2_split_kv_splits_for(num_reqs, num_kv_heads, max_blocks, window, d->sms);
}

int attn2_split_kv(const uint16_t *qkv, const uint16_t *kv_cache, int64_t num_pages,
                   const int32_t *block_table, int max_blocks, const int32_t *context_lens, int num_reqs,
                   int N, int num_kv_heads, int window, float scale, float eps, uint16_t *out, int splits,
                   void *workspace, size_t workspace_bytes, void *stream)
{
    int code;
    if (qkvf::check_attn2_args(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                               num_reqs, N, num_kv_heads, window, scale, eps, out, &code))
        return code;
    if (splits < 0 || splits > qkvf::kA2WsMaxSplits) return QKVF_ERR_VARIANT;
    if (num_reqs == 0) return QKVF_OK;
    if (!workspace) return QKVF_ERR_NULL;
    if (!qkvf::aligned(workspace, 256)) return QKVF_ERR_ALIGN;
    qkvf::DeviceState *d = nullptr;
    if (splits == 0) {   // the choice needs the device's SM count
        const int rc = qkvf::probe_device(&d);
        if (rc != QKVF_OK) return rc;
        splits = qkvf::attn2_split_kv_splits_for(num_reqs, num_kv_heads, max_blocks, window, d->sms);
    }
    const size_t need = qkvf::a2_workspace_bytes(num_reqs, num_kv_heads, splits);
    if (workspace_bytes < need) return QKVF_ERR_SIZES;
    const size_t out_b = (size_t)num_reqs * 8 * qkvf::kQPerKv * num_kv_heads * qkvf::kHeadDim * 2;
    const size_t qkv_b = (size_t)num_reqs * 8 * N * 2;
    const size_t cache_b = (size_t)num_pages * num_kv_heads * qkvf::kPageSlots * qkvf::kSlotWidth * 2;
    if (qkvf::overlap(workspace, need, out, out_b) || qkvf::overlap(workspace, need, qkv, qkv_b) ||
        qkvf::overlap(workspace, need, kv_cache, cache_b) ||
        qkvf::overlap(workspace, need, block_table, (size_t)num_reqs * max_blocks * 4) ||
        qkvf::overlap(workspace, need, context_lens, (size_t)num_reqs * 4))
        return QKVF_ERR_ARG;
    if (!d) {
        const int rc = qkvf::probe_device(&d);
        if (rc != QKVF_OK) return rc;
    }
    if (splits == 1)   // one CTA per (request, KV head) finishes its own rows: no partials to merge
        return qkvf::launch_attn2(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens, num_reqs,
                                  N, num_kv_heads, window, scale, eps, out, 1, nullptr, d->sms, stream);
    return qkvf::launch_attn2(qkv, kv_cache, num_pages, block_table, max_blocks, context_lens,
                              num_reqs, N, num_kv_heads, window, scale, eps, out, splits, workspace, d->sms, stream);
}

}  // extern "C"
