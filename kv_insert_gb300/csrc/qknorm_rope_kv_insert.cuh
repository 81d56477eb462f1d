// qknorm_rope_kv_insert: the unfused epilogue of the QKV projection, on its
// own, for any number of tokens (included by qkv_front.cu: one translation
// unit, one device status word).
//
// Source: fused_muse_spark_qknorm_rope_kv_insert, the kernel the fused front
// replaces (page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.
// attention.qkv_front", module docstring: the front writes what the
// projection GEMM followed by this kernel writes; page "...runtime.cute_ops",
// qkv_front paragraph).  On a BF16 projection output qkv [T, N] with rows
// [q | k | v | gate], in place: every q and k head is normed and rotated
// (the same arithmetic as the front's finish, qk_norm_rope_pair), v and gate
// heads are left as they are, and each token's k and v heads are written into
// its paged cache slot.  This is the path for token counts the fused front
// does not take (prefill, batches above 16).
//
// HBM-bound elementwise work: per token it reads the 9 nkv q/k heads and the
// nkv v heads (contiguous in the row: 1280 nkv bytes) and its cos|sin row,
// and writes the q/k heads back and 2 nkv slot halves.  With 16 KV heads or
// more a token is two work items (halves of its head groups), dealt round
// robin over the CTAs, so the busiest CTA holds at most half a token more
// than the average.  A
// producer warp copies each item's heads and table row into a shared-memory
// ring with 16-byte cp.async from its 32 lanes (up to ~100 KB in flight per
// CTA, two CTAs per SM; 48 KB and four CTAs per SM for 4 KV heads or fewer);
// consumer warps work from shared memory, 16 bytes per lane.
// (A bulk copy per token costs the SM's TMA unit ~0.2 us whatever its size,
// which set the pace at two copies per token; 32 lanes of cp.async do not.)

namespace qkvf {

struct EpiParams {
    uint16_t *qkv;
    const int64_t *positions;
    const int64_t *slots;
    const float *cos_sin;
    uint16_t *kv_cache;
    int64_t cos_rows;
    int64_t num_pages;
    unsigned long long wait_limit_ns;
    int T;
    int N;
    int nkv;
};

constexpr int kEpiMaxTokens = 1 << 24;
constexpr int kEpiMaxSlots = 24;

// The kernel's two shapes, by their consumer warps (warp 0 produces): two
// CTAs per SM with 8 consumer warps and 100 KB rings, the default; and for 4
// KV heads or fewer, where a token is 5 KB or less and the per-token steps
// (index loads, barriers) weigh most, four CTAs per SM with 4 consumer warps
// and 48 KB rings once there are more tokens than the default's CTAs (4096
// tokens at 1 / 2 / 4 KV heads: 9.30 -> 6.16, 9.87 -> 7.26, 11.49 -> 9.51
// us a call; with 8 or 16 KV heads no shape wins everywhere).
template <int kCW>
struct EpiShape {
    static constexpr int consumer_warps = kCW;
    static constexpr int threads = 32 * (kCW + 1);
    static constexpr int ctas_per_sm = kCW == 8 ? 2 : 4;
    static constexpr int ring_budget = kCW == 8 ? 100 * 1024 : 48 * 1024;   // the CTAs' rings fit one SM
    static_assert(kCW == 8 || kCW == 4, "two shapes");
};
constexpr int kEpiSmallNkv = 4;   // KV heads up to this take the four-CTA shape

__host__ __device__ inline int epi_groups(int nkv) { return ((kQPerKv + 2) * nkv + 7) >> 3; }

// Work items per token: with 16 or more 8-head groups (16 KV heads and up) a
// token is two items (its first ceil(groups / 2) groups, then the rest), so
// the busiest CTA holds at most half a token more than the average one;
// below that one item per token (halving then costs more in per-item
// barriers and index round trips than it saves: 8 KV heads at 4096 tokens
// 16.2 -> 20.9 us, at 16 KV heads and 8192 tokens 62.6 -> 59.5 us).
__host__ __device__ inline int epi_parts(int nkv) { return epi_groups(nkv) >= 16 ? 2 : 1; }

// the 8-head groups [lo, hi) of part `part` of a token
__host__ __device__ inline void epi_part_groups(int nkv, int part, int *lo, int *hi)
{
    const int g = epi_groups(nkv);
    if (epi_parts(nkv) == 1) {
        *lo = 0;
        *hi = g;
        return;
    }
    const int half = (g + 1) >> 1;
    *lo = part == 0 ? 0 : half;
    *hi = part == 0 ? half : g;
}

// bytes of one item's ring slot: its heads (all of the token's q | k | v
// region, or ceil(groups / 2) x 8 heads of it), its cos|sin row, and a
// 32-byte header (position, slot, flags), rounded to 128 bytes
__host__ __device__ inline uint32_t epi_part_bytes(int nkv)
{
    const int g = epi_groups(nkv);
    const int heads = (kQPerKv + 2) * nkv;
    return epi_parts(nkv) == 1 ? (uint32_t)heads * kHeadDim * 2 : (uint32_t)((g + 1) >> 1) * 8 * kHeadDim * 2;
}

__host__ __device__ inline uint32_t epi_slot_bytes(int nkv)
{
    return (epi_part_bytes(nkv) + kHeadDim * 4 + 32 + 127u) & ~127u;
}

__host__ __device__ inline int epi_slots(int nkv, int ring_budget)
{
    int n = ring_budget / (int)epi_slot_bytes(nkv);
    return n < 2 ? 2 : (n > kEpiMaxSlots ? kEpiMaxSlots : n);
}

__host__ __device__ inline uint32_t epi_smem_bytes(int nkv, int ring_budget)
{
    // slots, then full and empty barriers and the abort flag, plus alignment slack
    return (uint32_t)epi_slots(nkv, ring_budget) * epi_slot_bytes(nkv) + 2 * kEpiMaxSlots * 8 + 16 + 128;
}

// Packed FP32 pairs (Blackwell's f32x2 arithmetic): two IEEE round-to-nearest
// operations in one instruction, each lane's result the same bits as the
// scalar __fmul_rn / __fadd_rn / __fsub_rn.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Eight BF16 values (16 bytes: four rotation pairs 2j, 2j + 1) widened to
// FP32 and regrouped for packed arithmetic over pairs j and j + 1:
// ev[k] = (element 4k, element 4k + 2), od[k] = (element 4k + 1, element 4k + 3).
__device__ __forceinline__ void unpack8_pairs(const uint4 &v, uint64_t (&ev)[2], uint64_t (&od)[2])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        ev[k] = f2_pack(__uint_as_float(w[2 * k] << 16), __uint_as_float(w[2 * k + 1] << 16));
        od[k] = f2_pack(__uint_as_float(w[2 * k] & 0xFFFF0000u), __uint_as_float(w[2 * k + 1] & 0xFFFF0000u));
    }
}

// Sum of squares of one head held by 4 lanes, in exactly the association of
// the fused front's warp butterfly (qk_norm_rope_pair), so both kernels give
// the same bits.  In the front, lane l holds pair l (columns 2l, 2l+1) and the
// butterfly adds across lane bits 4, 3, 2, 1, 0 in that order.  Here lane c of
// the 4-lane group holds pairs 4c..4c+3 (lo) and 16+4c..16+4c+3 (hi): the
// front's lane bit 4 is lo/hi (added in registers), bits 3, 2 are this group's
// lane bits 1, 0 (two shuffle levels), and bits 1, 0 index the four pairs.
// Pair j's (x_2j^2 + x_2j+1^2) of lo and of hi, and their sum, are formed two
// pairs at a time.
__device__ __forceinline__ float head_sum_sq_front_order(const uint64_t (&lo_ev)[2], const uint64_t (&lo_od)[2],
                                                         const uint64_t (&hi_ev)[2], const uint64_t (&hi_od)[2])
{
    float a[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint64_t sl = f2_add(f2_mul(lo_ev[k], lo_ev[k]), f2_mul(lo_od[k], lo_od[k]));
        const uint64_t sh = f2_add(f2_mul(hi_ev[k], hi_ev[k]), f2_mul(hi_od[k], hi_od[k]));
        f2_unpack(f2_add(sl, sh), a[2 * k], a[2 * k + 1]);
    }
#pragma unroll
    for (int off = 2; off >= 1; off >>= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = __fadd_rn(a[j], __shfl_xor_sync(0xffffffffu, a[j], off));
    return __fadd_rn(__fadd_rn(a[0], a[2]), __fadd_rn(a[1], a[3]));
}

// Scale four rotation pairs by r and rotate them by (c, s), two pairs per
// packed operation: (a, b) = r (x_2j, x_2j+1); (a c - b s, b c + a s); BF16.
// cs points at cos[j0], sn at sin[j0] of the first pair (8-byte aligned).
__device__ __forceinline__ uint4 rope4_pairs(const uint64_t (&ev)[2], const uint64_t (&od)[2], uint64_t rr,
                                             const float *cs, const float *sn)
{
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint64_t c = *reinterpret_cast<const uint64_t *>(cs + 2 * k);
        const uint64_t s = *reinterpret_cast<const uint64_t *>(sn + 2 * k);
        const uint64_t a = f2_mul(ev[k], rr), b = f2_mul(od[k], rr);
        const uint64_t y0 = f2_sub(f2_mul(a, c), f2_mul(b, s));
        const uint64_t y1 = f2_add(f2_mul(b, c), f2_mul(a, s));
        float y00, y01, y10, y11;
        f2_unpack(y0, y00, y01);
        f2_unpack(y1, y10, y11);
        o[2 * k] = pack_bf16x2(__float2bfloat16_rn(y00), __float2bfloat16_rn(y10));
        o[2 * k + 1] = pack_bf16x2(__float2bfloat16_rn(y01), __float2bfloat16_rn(y11));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Work item u is part u % P of token u / P (P = epi_parts: the whole token,
// or its first ceil(groups / 2) 8-head groups and the rest); CTA b takes
// items b, b + G, b + 2G, ... (G = gridDim.x).  Warp 0 copies each item's heads (contiguous in the token's
// row) and its cos|sin row into a ring slot with 16-byte cp.async; warps
// 1..kCW take the item's heads in groups of 8 (lane l: head 8 g + l / 4,
// columns 8c..8c+7 and 32+8c..32+8c+7 with c = l % 4), norm and rotate q / k
// heads in place in global memory and write k / v heads into the cache slot.
template <int kCW>
__global__ void __launch_bounds__(EpiShape<kCW>::threads, EpiShape<kCW>::ctas_per_sm)
    qknorm_rope_kv_insert_kernel(const EpiParams p)
{
    constexpr int kEpiConsumerWarps = kCW;
    extern __shared__ uint8_t epi_smem_dyn[];
    uint8_t *smem = epi_smem_dyn + ((128u - (smem_u32(epi_smem_dyn) & 127u)) & 127u);
    const int nkv = p.nkv;
    const uint32_t slot_bytes = epi_slot_bytes(nkv);
    const int nslots = epi_slots(nkv, EpiShape<kCW>::ring_budget);
    const uint32_t region = epi_part_bytes(nkv);   // the cos|sin row follows an item's heads
    const int parts = epi_parts(nkv);
    const int64_t U = (int64_t)p.T * parts;        // work items
    const uint32_t full0 = smem_u32(smem + nslots * slot_bytes);
    const uint32_t empty0 = full0 + 8 * kEpiMaxSlots;
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + nslots * slot_bytes + 16 * kEpiMaxSlots);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int q_heads = kQPerKv * nkv, qk_heads = q_heads + nkv, heads = qk_heads + nkv;
    const int64_t slot_end = p.num_pages * (int64_t)kPageSlots;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nslots; ++s) {
            // the 32 lanes' copies land (32) and lane 0's header (1)
            mbar_init(full0 + 8 * s, 33);
            mbar_init(empty0 + 8 * s, kEpiConsumerWarps);   // one arrival per consumer warp
        }
        *s_abort = 0;
        fence_barrier_init();
        griddep_launch_dependents();
    }
    __syncthreads();
    griddep_wait();   // qkv, indices and table are written by the kernels before this one

    if (warp == 0) {
        // ---- produce: 32 items' indices per warp load, then each item's copies ----
        // An item's heads need no index, so their copy is issued before the
        // index loads are first used: the data and the indices come in side
        // by side.
        unsigned bad = 0u;
        int i = 0;
        bool stop = false;
        for (int64_t ub = blockIdx.x; ub < U && !stop; ub += 32 * G) {
            const int64_t ul = ub + lane * G, tl = ul / parts;
            int64_t pos_l = -1, slot_l = -1;
            if (ul < U) {
                pos_l = p.positions[tl];
                slot_l = p.slots[tl];
            }
            for (int j = 0; j < 32; ++j, ++i) {
                const int64_t u = ub + j * G, t = u / parts;
                if (u >= U) break;   // the same for every lane
                int g_lo, g_hi;
                epi_part_groups(nkv, (int)(u % parts), &g_lo, &g_hi);
                const int h_end = 8 * g_hi < heads ? 8 * g_hi : heads;
                const uint32_t bytes = (uint32_t)(h_end - 8 * g_lo) * kHeadDim * 2;
                const int s = i % nslots, use = i / nslots;
                int ok = 1;
                if (lane == 0 && use > 0)
                    ok = bounded_wait(empty0 + 8 * s, (uint32_t)((use - 1) & 1), s_abort, p.wait_limit_ns, true);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    stop = true;
                    break;
                }
                uint8_t *base = smem + (size_t)s * slot_bytes;
                const uint32_t bar = full0 + 8 * s;
                const uint8_t *src =
                    reinterpret_cast<const uint8_t *>(p.qkv + (size_t)t * p.N + (size_t)8 * g_lo * kHeadDim);
                for (uint32_t c = (uint32_t)lane; c < bytes / 16; c += 32)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(base) + 16 * c),
                                 "l"(src + 16 * c)
                                 : "memory");
                const int64_t pos = __shfl_sync(0xffffffffu, pos_l, j);
                const int64_t sl = __shfl_sync(0xffffffffu, slot_l, j);
                const bool pos_ok = pos >= 0 && pos < p.cos_rows;
                const bool ins = sl >= 0 && sl < slot_end && pos_ok;
                if (lane == 0) {
                    int64_t *hdr = reinterpret_cast<int64_t *>(base + region + kHeadDim * 4);
                    hdr[0] = pos;
                    hdr[1] = sl;
                    hdr[2] = (pos_ok ? 1 : 0) | (ins ? 2 : 0);
                }
                if (pos_ok && lane < kHeadDim * 4 / 16)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(base + region) + 16 * lane),
                                 "l"(reinterpret_cast<const uint8_t *>(p.cos_sin + pos * kHeadDim) + 16 * lane)
                                 : "memory");
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
                if (lane == 0) mbar_arrive(bar);   // the header
            }
            if (ul < U)
                bad |= (pos_l >= 0 && pos_l < p.cos_rows ? 0u : QKVF_STATUS_BAD_POSITION) |
                       (slot_l >= slot_end ? QKVF_STATUS_BAD_SLOT : 0u);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // nothing of ours left in flight
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0 && bad != 0u) atomicOr(&g_status, bad);
    } else {
        // ---- consume: groups of 8 heads, 4 lanes x 32 bytes per head ------
        // The CTA's (item, group) pairs are dealt round robin over the consumer
        // warps across item boundaries, so an item with fewer groups than warps
        // does not leave warps idle.  Every warp waits on every item in order
        // (the barrier parity never runs more than one phase ahead) and arrives
        // once on the item's empty barrier after its groups of the item.
        const int cw = warp - 1, sub = lane >> 2, part = lane & 3;
        int i = 0;
        int64_t first = 0;   // (item, group) index of this item's first group
        for (int64_t u = blockIdx.x; u < U; u += G, ++i) {
            const int64_t t = u / parts;
            int g_lo, g_hi;
            epi_part_groups(nkv, (int)(u % parts), &g_lo, &g_hi);
            const int s = i % nslots;
            const int g0 = g_lo + (int)(((int64_t)cw - first % kEpiConsumerWarps + kEpiConsumerWarps) %
                                        kEpiConsumerWarps);
            first += g_hi - g_lo;
            const bool landed = mbar_try_wait(full0 + 8 * s, (uint32_t)((i / nslots) & 1)) ||
                                bounded_wait(full0 + 8 * s, (uint32_t)((i / nslots) & 1), s_abort,
                                             p.wait_limit_ns, true);
            if (__all_sync(0xffffffffu, landed)) {
                const uint8_t *base = smem + (size_t)s * slot_bytes;
                const int64_t *hdr = reinterpret_cast<const int64_t *>(base + region + kHeadDim * 4);
                const int64_t sl = hdr[1];
                const int flags = (int)hdr[2];
                const bool pos_ok = flags & 1, ins = flags & 2;
                const float *row = reinterpret_cast<const float *>(base + region);
                uint16_t *qrow = p.qkv + (size_t)t * p.N + 8 * part;
                uint16_t *crow = nullptr;
                if (ins) {
                    const int64_t page = sl / kPageSlots, offs = sl % kPageSlots;
                    crow = p.kv_cache + ((page * nkv) * kPageSlots + offs) * kSlotWidth + 8 * part;
                }
                for (int grp = g0; grp < g_hi; grp += kEpiConsumerWarps) {
                    // lane: head 8 grp + l / 4; bytes 16 c and 64 + 16 c of the head (c = l % 4)
                    const int h = grp * 8 + sub;
                    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
                    if (h < heads) {
                        const uint8_t *src = base + (h - 8 * g_lo) * (kHeadDim * 2) + 16 * part;
                        v0 = *reinterpret_cast<const uint4 *>(src);
                        v1 = *reinterpret_cast<const uint4 *>(src + 64);
                    }
                    if (grp * 8 < qk_heads && pos_ok) {   // the whole warp: shuffles inside
                        uint64_t lo_ev[2], lo_od[2], hi_ev[2], hi_od[2];
                        unpack8_pairs(v0, lo_ev, lo_od);
                        unpack8_pairs(v1, hi_ev, hi_od);
                        const float ss = head_sum_sq_front_order(lo_ev, lo_od, hi_ev, hi_od);
                        const float ms = __fmul_rn(ss, 1.0f / (float)kHeadDim);   // exact: a power of two
                        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, kEps)));
                        const uint64_t rr = f2_pack(r, r);
                        const uint4 o0 = rope4_pairs(lo_ev, lo_od, rr, row + 4 * part, row + 32 + 4 * part);
                        const uint4 o1 = rope4_pairs(hi_ev, hi_od, rr, row + 16 + 4 * part, row + 48 + 4 * part);
                        if (h < qk_heads) {
                            v0 = o0;
                            v1 = o1;
                            uint16_t *dst = qrow + (size_t)h * kHeadDim;
                            *reinterpret_cast<uint4 *>(dst) = v0;
                            *reinterpret_cast<uint4 *>(dst + 32) = v1;
                        }
                    }
                    if (h >= q_heads && h < heads && ins) {   // k or v head of an inserting token
                        const bool is_v = h >= qk_heads;
                        const int gkv = h - q_heads - (is_v ? nkv : 0);
                        uint16_t *dst = crow + (size_t)gkv * kPageSlots * kSlotWidth + (is_v ? kHeadDim : 0);
                        *reinterpret_cast<uint4 *>(dst) = v0;
                        *reinterpret_cast<uint4 *>(dst + 32) = v1;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
    }
}

const char *check_epi_args(uint16_t *qkv, const int64_t *positions, const int64_t *slots,
                           const float *cos_sin, int64_t cos_sin_rows, uint16_t *kv_cache,
                           int64_t num_pages, int T, int N, int num_kv_heads, int *code)
{
    *code = QKVF_ERR_TOKENS;
    if (T < 0 || T > kEpiMaxTokens) return "T must be 0..16777216 tokens";
    *code = QKVF_ERR_SHAPE;
    if (num_kv_heads < 1 || num_kv_heads > 64) return "num_kv_heads must be 1..64";
    if (N != 2 * (kQPerKv + 1) * kHeadDim * num_kv_heads)
        return "N must be 1152 * num_kv_heads: rows [q | k | v | gate], 8 q and 8 gate heads of 64 per KV head";
    *code = QKVF_ERR_SIZES;
    if (cos_sin_rows < 1 || cos_sin_rows > (int64_t(1) << 40)) return "cos_sin_rows must be >= 1";
    if (num_pages < 1 || num_pages > (int64_t(1) << 36)) return "num_pages must be >= 1";
    *code = QKVF_OK;
    if (T == 0) return nullptr;
    *code = QKVF_ERR_NULL;
    if (!qkv || !positions || !slots || !cos_sin || !kv_cache) return "a required pointer is NULL";
    *code = QKVF_ERR_ALIGN;
    if (!aligned(qkv, 16) || !aligned(kv_cache, 16) || !aligned(cos_sin, 16))
        return "qkv, kv_cache and cos_sin must be 16-byte aligned";
    if (!aligned(positions, 8) || !aligned(slots, 8))
        return "positions and slots must be 8-byte aligned int64";
    *code = QKVF_ERR_ARG;
    const size_t qkv_b = (size_t)T * N * 2;
    const size_t cache_b = (size_t)num_pages * num_kv_heads * kPageSlots * kSlotWidth * 2;
    const size_t cs_b = (size_t)cos_sin_rows * kHeadDim * 4, idx_b = (size_t)T * 8;
    const void *ins[] = {cos_sin, positions, slots};
    const size_t in_b[] = {cs_b, idx_b, idx_b};
    for (int i = 0; i < 3; ++i)
        if (overlap(ins[i], in_b[i], qkv, qkv_b) || overlap(ins[i], in_b[i], kv_cache, cache_b))
            return "an input overlaps qkv or kv_cache";
    if (overlap(qkv, qkv_b, kv_cache, cache_b)) return "qkv overlaps kv_cache";
    *code = QKVF_OK;
    return nullptr;
}

bool prepare_epi_kernel()
{
    // each shape's largest ring over the KV head counts it takes
    uint32_t most8 = 0, most4 = 0;
    for (int nkv = kEpiSmallNkv + 1; nkv <= 64; ++nkv) {
        const uint32_t b = epi_smem_bytes(nkv, EpiShape<8>::ring_budget);
        most8 = b > most8 ? b : most8;
    }
    for (int nkv = 1; nkv <= kEpiSmallNkv; ++nkv) {
        const uint32_t b = epi_smem_bytes(nkv, EpiShape<4>::ring_budget);
        most4 = b > most4 ? b : most4;
    }
    return cudaFuncSetAttribute((const void *)qknorm_rope_kv_insert_kernel<8>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most8) == cudaSuccess &&
           cudaFuncSetAttribute((const void *)qknorm_rope_kv_insert_kernel<4>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most4) == cudaSuccess;
}

int launch_epi(uint16_t *qkv, const int64_t *positions, const int64_t *slots, const float *cos_sin,
               int64_t cos_sin_rows, uint16_t *kv_cache, int64_t num_pages, int T, int N,
               int num_kv_heads, int sms, void *stream)
{
    EpiParams prm;
    prm.qkv = qkv;
    prm.positions = positions;
    prm.slots = slots;
    prm.cos_sin = cos_sin;
    prm.kv_cache = kv_cache;
    prm.cos_rows = cos_sin_rows;
    prm.num_pages = num_pages;
    prm.T = T;
    prm.N = N;
    prm.nkv = num_kv_heads;
    prm.wait_limit_ns = g_wait_limit_ns;
    // the four-CTA shape once the default's CTAs would hold more than one
    // item each (below that a token's groups spread over 8 warps finish sooner)
    const bool small = num_kv_heads <= kEpiSmallNkv &&
                       (int64_t)T * epi_parts(num_kv_heads) > (int64_t)sms * EpiShape<8>::ctas_per_sm;
    const int per_sm = small ? EpiShape<4>::ctas_per_sm : EpiShape<8>::ctas_per_sm;
    int64_t blocks = (int64_t)sms * per_sm;   // CTAs per SM, each walking its items
    if (blocks > (int64_t)T * epi_parts(num_kv_heads)) blocks = (int64_t)T * epi_parts(num_kv_heads);
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(small ? EpiShape<4>::threads : EpiShape<8>::threads, 1, 1);
    cfg.dynamicSmemBytes =
        epi_smem_bytes(num_kv_heads, small ? EpiShape<4>::ring_budget : EpiShape<8>::ring_budget);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = small ? cudaLaunchKernelEx(&cfg, qknorm_rope_kv_insert_kernel<4>, prm)
                                : cudaLaunchKernelEx(&cfg, qknorm_rope_kv_insert_kernel<8>, prm);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return QKVF_ERR_CUDA;
    }
    return QKVF_OK;
}

}  // namespace qkvf

extern "C" {

const char *qknorm_rope_kv_insert_unsupported(uint16_t *qkv, const int64_t *positions,
                                              const int64_t *slots, const float *cos_sin,
                                              int64_t cos_sin_rows, uint16_t *kv_cache,
                                              int64_t num_pages, int T, int N, int num_kv_heads)
{
    int code;
    const char *why = qkvf::check_epi_args(qkv, positions, slots, cos_sin, cos_sin_rows, kv_cache,
                                           num_pages, T, N, num_kv_heads, &code);
    if (why) return why;
    qkvf::DeviceState *d;
    const int rc = qkvf::probe_device(&d);
    return rc == QKVF_OK ? nullptr : qkv_front_strerror(rc);
}

int qknorm_rope_kv_insert(uint16_t *qkv, const int64_t *positions, const int64_t *slots,
                          const float *cos_sin, int64_t cos_sin_rows, uint16_t *kv_cache,
                          int64_t num_pages, int T, int N, int num_kv_heads, void *stream)
{
    int code;
    if (qkvf::check_epi_args(qkv, positions, slots, cos_sin, cos_sin_rows, kv_cache, num_pages, T,
                             N, num_kv_heads, &code))
        return code;
    if (T == 0) return QKVF_OK;
    qkvf::DeviceState *d;
    const int rc = qkvf::probe_device(&d);
    if (rc != QKVF_OK) return rc;
    return qkvf::launch_epi(qkv, positions, slots, cos_sin, cos_sin_rows, kv_cache, num_pages, T, N,
                            num_kv_heads, d->sms, stream);
}

}  // extern "C"
