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
// nkv v heads (128 B each) and writes the q/k heads back and 2 nkv slot
// halves.  One warp per task of 4 heads of a token, 16 bytes per lane; tasks
// are dealt to warps kEpiUnroll at a time and the loads of a round are issued
// before any is used (head values first, then indices, then table rows), so
// each warp keeps several 512-byte requests in flight.

namespace qkvf {

struct EpiParams {
    uint16_t *qkv;
    const int64_t *positions;
    const int64_t *slots;
    const float *cos_sin;
    uint16_t *kv_cache;
    int64_t cos_rows;
    int64_t num_pages;
    int T;
    int N;
    int nkv;
};

constexpr int kEpiThreads = 256;
constexpr int kEpiUnroll = 3;            // head groups per warp per round, loads issued first
constexpr int kEpiMaxTokens = 1 << 24;

// Sum of squares of one head held as 8 lanes x 8 values, in exactly the
// association of the fused front's warp butterfly (qk_norm_rope_pair), so
// both kernels give the same bits.  In the front, lane l holds columns
// (2l, 2l+1) and the butterfly adds across lane bits 4, 3, 2, then 1, 0.  Here
// lane c of the group holds columns 8c..8c+7, i.e. the front's lanes 4c..4c+3:
// the front's lane bits 4, 3, 2 are this group's lane bits 2, 1, 0, and its
// bits 1, 0 are the four pairs inside this lane.
__device__ __forceinline__ float head_sum_sq_front_order(const float (&f)[8])
{
    float s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        s[j] = __fadd_rn(__fmul_rn(f[2 * j], f[2 * j]), __fmul_rn(f[2 * j + 1], f[2 * j + 1]));
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j] = __fadd_rn(s[j], __shfl_xor_sync(0xffffffffu, s[j], off));
    return __fadd_rn(__fadd_rn(s[0], s[2]), __fadd_rn(s[1], s[3]));
}

// One warp per task of 4 consecutive heads of one token (q, k or v heads;
// gate heads need nothing): lane l handles head 4 g + l / 8, columns
// 8 (l % 8) .. 8 (l % 8) + 7, as one 16-byte access.
__global__ void __launch_bounds__(kEpiThreads, 3) qknorm_rope_kv_insert_kernel(const EpiParams p)
{
    griddep_wait();   // qkv, indices and table are written by the kernels before this one
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3, chunk = lane & 7;
    const int64_t warp_id = ((int64_t)blockIdx.x * kEpiThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kEpiThreads) >> 5;
    const int q_heads = kQPerKv * p.nkv;
    const int qk_heads = q_heads + p.nkv;
    const int heads = qk_heads + p.nkv;          // q, k and v heads
    const int groups = (heads + 3) >> 2;         // per token
    const int64_t total = (int64_t)p.T * groups;
    const int64_t slot_end = p.num_pages * (int64_t)kPageSlots;
    unsigned bad = 0u;

    for (int64_t base = warp_id * kEpiUnroll; base < total; base += nwarps * kEpiUnroll) {
        int tok[kEpiUnroll], head[kEpiUnroll];
        uint4 val[kEpiUnroll];
        int64_t pos[kEpiUnroll], slot[kEpiUnroll];
        float4 cv[kEpiUnroll], sv[kEpiUnroll];
        // the head values first: they depend on nothing
#pragma unroll
        for (int u = 0; u < kEpiUnroll; ++u) {
            const int64_t task = base + u;
            const bool in = task < total;
            tok[u] = in ? (int)(task / groups) : 0;
            head[u] = in ? (int)(task % groups) * 4 + sub : heads;   // heads: nothing to do
            val[u] = make_uint4(0u, 0u, 0u, 0u);
            if (head[u] < heads)
                val[u] = *reinterpret_cast<const uint4 *>(p.qkv + (size_t)tok[u] * p.N +
                                                          (size_t)head[u] * kHeadDim + 8 * chunk);
        }
#pragma unroll
        for (int u = 0; u < kEpiUnroll; ++u) {
            pos[u] = -1;
            slot[u] = -1;
            if (base + u < total) {
                pos[u] = p.positions[tok[u]];
                slot[u] = p.slots[tok[u]];
            }
        }
#pragma unroll
        for (int u = 0; u < kEpiUnroll; ++u) {
            cv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            sv[u] = cv[u];
            const bool pos_ok = pos[u] >= 0 && pos[u] < p.cos_rows;
            if (head[u] < qk_heads && pos_ok) {
                const float *row = p.cos_sin + pos[u] * kHeadDim;
                cv[u] = *reinterpret_cast<const float4 *>(row + 4 * chunk);
                sv[u] = *reinterpret_cast<const float4 *>(row + 32 + 4 * chunk);
            }
        }
#pragma unroll
        for (int u = 0; u < kEpiUnroll; ++u) {
            if (base + u >= total) continue;   // the same for every lane of the warp
            const bool pos_ok = pos[u] >= 0 && pos[u] < p.cos_rows;
            const bool ins = slot[u] >= 0 && slot[u] < slot_end && pos_ok;
            if (head[u] == 0)
                bad |= (pos_ok ? 0u : QKVF_STATUS_BAD_POSITION) |
                       (slot[u] >= slot_end ? QKVF_STATUS_BAD_SLOT : 0u);
            const int h = head[u];
            uint4 word = val[u];
            // q / k heads of the group: the whole warp runs the shuffles (lanes of
            // v heads or of heads past the last one compute values they drop)
            const bool qk_group = (h - sub) < qk_heads;   // the group's first head
            if (qk_group && pos_ok) {
                const uint32_t w4[4] = {val[u].x, val[u].y, val[u].z, val[u].w};
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&w4[j]);
                    f[2 * j] = __low2float(pr);
                    f[2 * j + 1] = __high2float(pr);
                }
                const float ss = head_sum_sq_front_order(f);
                const float ms = __fdiv_rn(ss, (float)kHeadDim);
                const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, kEps)));
                const float cc[4] = {cv[u].x, cv[u].y, cv[u].z, cv[u].w};
                const float ss4[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = __fmul_rn(f[2 * j], r), b = __fmul_rn(f[2 * j + 1], r);
                    const float y0 = __fsub_rn(__fmul_rn(a, cc[j]), __fmul_rn(b, ss4[j]));
                    const float y1 = __fadd_rn(__fmul_rn(b, cc[j]), __fmul_rn(a, ss4[j]));
                    o[j] = pack_bf16x2(__float2bfloat16_rn(y0), __float2bfloat16_rn(y1));
                }
                if (h < qk_heads) {
                    word = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(p.qkv + (size_t)tok[u] * p.N + (size_t)h * kHeadDim +
                                               8 * chunk) = word;
                }
            }
            if (h >= q_heads && h < heads && ins && (h >= qk_heads || pos_ok)) {
                const bool is_v = h >= qk_heads;
                const int gkv = h - q_heads - (is_v ? p.nkv : 0);
                const int64_t page = slot[u] / kPageSlots, offs = slot[u] % kPageSlots;
                uint16_t *dst = p.kv_cache + ((page * p.nkv + gkv) * kPageSlots + offs) * kSlotWidth +
                                (is_v ? kHeadDim : 0) + 8 * chunk;
                *reinterpret_cast<uint4 *>(dst) = word;
            }
        }
    }
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0 && bad != 0u) atomicOr(&g_status, bad);
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
    const int64_t tasks = (int64_t)T * (((kQPerKv + 2) * num_kv_heads + 3) / 4);
    const int64_t warps_needed = (tasks + kEpiUnroll - 1) / kEpiUnroll;
    int64_t blocks = (warps_needed + (kEpiThreads / 32) - 1) / (kEpiThreads / 32);
    const int64_t resident = (int64_t)sms * 3;   // one full wave at 3 blocks per SM
    if (blocks > resident) blocks = resident;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(kEpiThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, qknorm_rope_kv_insert_kernel, prm) != cudaSuccess) {
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
