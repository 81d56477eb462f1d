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
// halves.  One warp per (token, head) task; lane l owns the pair (2l, 2l+1).
// Tasks are dealt to warps kEpiUnroll at a time and the loads of a chunk are
// all issued before any is used, so each warp keeps several 128-B requests in
// flight.

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
constexpr int kEpiUnroll = 4;
constexpr int kEpiMaxTokens = 1 << 24;

__global__ void __launch_bounds__(kEpiThreads, 4) qknorm_rope_kv_insert_kernel(const EpiParams p)
{
    griddep_wait();   // qkv, indices and table are written by the kernels before this one
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = ((int64_t)blockIdx.x * kEpiThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kEpiThreads) >> 5;
    const int q_heads = kQPerKv * p.nkv;
    const int qk_heads = q_heads + p.nkv;
    const int per_token = qk_heads + p.nkv;   // q, k and v heads; gate heads need nothing
    const int64_t total = (int64_t)p.T * per_token;
    const int64_t slot_end = p.num_pages * (int64_t)kPageSlots;
    unsigned bad = 0u;

    for (int64_t base = warp_id * kEpiUnroll; base < total; base += nwarps * kEpiUnroll) {
        uint32_t val[kEpiUnroll];
        float c[kEpiUnroll], sn[kEpiUnroll];
        int64_t slot[kEpiUnroll];
        int tok[kEpiUnroll], head[kEpiUnroll], flag[kEpiUnroll];
#pragma unroll
        for (int u = 0; u < kEpiUnroll; ++u) {
            const int64_t task = base + u;
            flag[u] = 0;   // bit 0: a task; bit 1: position in range; bit 2: insert
            tok[u] = 0;
            head[u] = 0;
            slot[u] = -1;
            val[u] = 0u;
            c[u] = 0.f;
            sn[u] = 0.f;
            if (task < total) {
                const int t = (int)(task / per_token);
                const int h = (int)(task % per_token);
                const int64_t pos = p.positions[t];
                const int64_t sl = p.slots[t];
                const bool pos_ok = pos >= 0 && pos < p.cos_rows;
                const bool ins = sl >= 0 && sl < slot_end && pos_ok;
                tok[u] = t;
                head[u] = h;
                slot[u] = sl;
                flag[u] = 1 | (pos_ok ? 2 : 0) | (ins ? 4 : 0);
                if (h == 0)
                    bad |= (pos_ok ? 0u : QKVF_STATUS_BAD_POSITION) |
                           (sl >= slot_end ? QKVF_STATUS_BAD_SLOT : 0u);
                val[u] = reinterpret_cast<const uint32_t *>(p.qkv + (size_t)t * p.N +
                                                            (size_t)h * kHeadDim)[lane];
                if (h < qk_heads && pos_ok) {
                    const float *row = p.cos_sin + pos * kHeadDim;
                    c[u] = row[lane];
                    sn[u] = row[32 + lane];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kEpiUnroll; ++u) {
            if (!(flag[u] & 1)) continue;   // the same for every lane of the warp
            const int h = head[u];
            uint32_t word = val[u];
            if (h < qk_heads) {
                if (!(flag[u] & 2)) continue;   // no table row: the head is left as it was
                const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&val[u]);
                word = qk_norm_rope_pair(__low2float(pr), __high2float(pr), c[u], sn[u]);
                reinterpret_cast<uint32_t *>(p.qkv + (size_t)tok[u] * p.N +
                                             (size_t)h * kHeadDim)[lane] = word;
            }
            if (h >= q_heads && (flag[u] & 4)) {   // k or v head of an inserting token
                const bool is_v = h >= qk_heads;
                const int gkv = h - q_heads - (is_v ? p.nkv : 0);
                const int64_t page = slot[u] / kPageSlots, offs = slot[u] % kPageSlots;
                uint16_t *dst = p.kv_cache + ((page * p.nkv + gkv) * kPageSlots + offs) * kSlotWidth +
                                (is_v ? kHeadDim : 0);
                reinterpret_cast<uint32_t *>(dst)[lane] = word;
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
    const int64_t tasks = (int64_t)T * (kQPerKv + 2) * num_kv_heads;
    const int64_t warps_needed = (tasks + kEpiUnroll - 1) / kEpiUnroll;
    int64_t blocks = (warps_needed + (kEpiThreads / 32) - 1) / (kEpiThreads / 32);
    const int64_t resident = (int64_t)sms * 4;   // one full wave at 4 blocks per SM
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
