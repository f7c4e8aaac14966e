// fa2_bwd.cu -- host-side launch of the backward pass ("Chapter 08: Flash
// Attention -- blocked attention", section 6): the Delta kernel, then dQ (query
// tiles resident), then dK and dV (key/value tiles resident), all on one stream.
#include <atomic>

#include "fa2_bwd_kernel.cuh"
#include "fa2_launch.cuh"

namespace fa2 {

// dK/dV: 128 keys resident, query tiles of 64 streamed through a 4-stage ring
// (dV, dK and two 64-column score pairs fill TMEM at D = 128, where K and V stay in
// shared memory; at D = 64 K and V are also copied into TMEM as the score products' A
// operands);
// dQ: 128 queries resident, key tiles of 64 through a 4-stage ring.  Two score
// buffer pairs let one step's MMAs run while the previous step's elementwise
// work finishes.
//
// D = 256: two CTAs per resident tile, each accumulating 128 of the 256 gradient
// columns (both compute the step's full score products).  The resident tiles take
// 2 x 64 KB of shared memory, so the streamed tiles are 32 rows (16 KB each) through a
// 3-stage ring, with one elementwise warp per lane quarter.  The 32-column score
// buffers leave TMEM room for Q and dO (dQ kernel) and for K (dK/dV kernel) as the A
// operands of the score products.
template <int D>
using BwdKV = BwdCfg<D, 128, (D == 256 ? 32 : 64), (D == 256 ? 3 : 4), (D == 256 ? 4 : 8), (D == 256 ? 128 : D)>;
template <int D>
using BwdQ = BwdCfg<D, 128, (D == 256 ? 32 : 64), (D == 256 ? 3 : 4), (D == 256 ? 4 : 8), (D == 256 ? 128 : D)>;
static_assert(BWD_STAT_TILE_ROWS == BWD_STAT_ROWS, "workspace sizing and kernels agree on the statistics tiles");

template <class K>
static bool set_smem(K kernel, int bytes, int device, std::atomic<unsigned long long> &configured)
{
    const unsigned long long bit = (device >= 0 && device < 64) ? (1ull << device) : 0ull;
    if (bit && (configured.load() & bit))
        return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    configured.fetch_or(bit);
    return true;
}

// A [B, H, L, D] view as a tensor map with boxes of 64 columns by box_rows rows of one
// head: 3-D (D, L, B*H) when its batch stride is H times its head stride (or B == 1),
// else 4-D (D, L, H, B).  Sets *is3 accordingly.
static bool encode_bwd_map(EncodeTiledFn encode, CUtensorMap *m, const void *ptr, int D, int L, int H, int B,
                           BhlStrides st, int box_rows, bool *is3)
{
    *is3 = B == 1 || st.b == st.h * H;
    if (!*is3)
        return encode_bhld_strided(encode, m, ptr, D, L, H, B, st, box_rows);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                          static_cast<cuuint64_t>(B) * static_cast<cuuint64_t>(H)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(st.l) * 2, static_cast<cuuint64_t>(st.h) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static fa2_status launch_bwd_d(const BwdArgs &a)
{
    using CKV = BwdKV<D>;
    using CQ = BwdQ<D>;
    const int BH = a.B * a.H;
    // every input as a tensor map built from its strides (3-D where the heads collapse)
    CUtensorMap q_res, do_res, k_str, v_str, k_res, v_res, q_str, do_str;
    bool q3, k3, v3, do3;
    if (!encode_bwd_map(a.encode, &q_res, a.q, D, a.Lq, a.H, a.B, a.sq, CQ::RES, &q3) ||
        !encode_bwd_map(a.encode, &do_res, a.dout, D, a.Lq, a.H, a.B, a.sdo, CQ::RES, &do3) ||
        !encode_bwd_map(a.encode, &k_str, a.k, D, a.Lk, a.H, a.B, a.sk, CQ::STR, &k3) ||
        !encode_bwd_map(a.encode, &v_str, a.v, D, a.Lk, a.H, a.B, a.sv, CQ::STR, &v3) ||
        !encode_bwd_map(a.encode, &k_res, a.k, D, a.Lk, a.H, a.B, a.sk, CKV::RES, &k3) ||
        !encode_bwd_map(a.encode, &v_res, a.v, D, a.Lk, a.H, a.B, a.sv, CKV::RES, &v3) ||
        !encode_bwd_map(a.encode, &q_str, a.q, D, a.Lq, a.H, a.B, a.sq, CKV::STR, &q3) ||
        !encode_bwd_map(a.encode, &do_str, a.dout, D, a.Lq, a.H, a.B, a.sdo, CKV::STR, &do3))
        return FA2_ERR_CUDA;
    BwdParams p;
    const int n_stat_tiles = (a.Lq + BWD_STAT_ROWS - 1) / BWD_STAT_ROWS;
    p.stats = a.stats;
    p.n_stat_tiles = n_stat_tiles;
    p.dq = static_cast<uint16_t *>(a.dq);
    p.dk = static_cast<uint16_t *>(a.dk);
    p.dv = static_cast<uint16_t *>(a.dv);
    p.dq_sb = a.sdq.b;
    p.dq_sh = a.sdq.h;
    p.dq_sl = a.sdq.l;
    p.dk_sb = a.sdk.b;
    p.dk_sh = a.sdk.h;
    p.dk_sl = a.sdk.l;
    p.dv_sb = a.sdv.b;
    p.dv_sh = a.sdv.h;
    p.dv_sl = a.sdv.l;
    p.H = a.H;
    // Causal grids: when every head's streamed tiles (Q and dO, or K and V) together fit in
    // half of L2, one group of all heads (plain heaviest-first order); otherwise groups of
    // as many heads as fit in a quarter of L2.  Measured on B1 H32 L16384 D128 (256 MB of
    // streamed tiles): 1098-1112 -> 1182 TFLOP/s causal; splitting c3's 64 MB into groups
    // of 16 heads cost 1-2 %.
    {
        const long long per_head = 2ll * (a.Lq > a.Lk ? a.Lq : a.Lk) * D * 2;
        long long g = BH;
        if (per_head * BH > (64ll << 20))
            g = (32ll << 20) / per_head;
        p.head_group = static_cast<int>(g < 1 ? 1 : g > BH ? BH : g);
    }
    p.maps3 = (q3 ? 1 << BWD_MAP_Q : 0) | (k3 ? 1 << BWD_MAP_K : 0) | (v3 ? 1 << BWD_MAP_V : 0) |
              (do3 ? 1 << BWD_MAP_DO : 0);
    p.err = a.err;
    p.wait_limit_ns = a.wait_limit_ns;
    p.Lq = a.Lq;
    p.Lk = a.Lk;
    p.BH = BH;
    p.causal = a.causal ? 1 : 0;
    p.window = a.causal ? a.window : -1;
    p.scale = a.scale;
    p.scale_log2 = a.scale * BWD_LOG2E;

    static std::atomic<unsigned long long> cfg_q{0}, cfg_kv{0};
    if (!set_smem(fa2_bwd_q_kernel<CQ>, CQ::SMEM_BYTES, a.device, cfg_q) ||
        !set_smem(fa2_bwd_kv_kernel<CKV>, CKV::SMEM_BYTES, a.device, cfg_kv))
        return FA2_ERR_CUDA;
    if (a.Lq > 0) {
        const long long rows = static_cast<long long>(BH) * n_stat_tiles * BWD_STAT_ROWS;
        constexpr int rpb = bwd_delta_rows_per_block<D>();
        fa2_bwd_delta_kernel<D><<<static_cast<unsigned>((rows + rpb - 1) / rpb), BWD_DELTA_THREADS, 0, a.stream>>>(
            static_cast<const uint16_t *>(a.o), static_cast<const uint16_t *>(a.dout), a.lse, a.stats, a.Lq,
            n_stat_tiles, rows, a.H, BwdRowStrides{a.so.b, a.so.h, a.so.l}, BwdRowStrides{a.sdo.b, a.sdo.h, a.sdo.l});
        const long long n_qt = (a.Lq + CQ::RES - 1) / CQ::RES;
        fa2_bwd_q_kernel<CQ><<<static_cast<unsigned>(n_qt * BH * CQ::NH), CQ::NUM_THREADS, CQ::SMEM_BYTES,
                               a.stream>>>(q_res, do_res, k_str, v_str, p);
    }
    const long long n_kt = (a.Lk + CKV::RES - 1) / CKV::RES;
    fa2_bwd_kv_kernel<CKV><<<static_cast<unsigned>(n_kt * BH * CKV::NH), CKV::NUM_THREADS, CKV::SMEM_BYTES,
                             a.stream>>>(k_res, v_res, q_str, do_str, p);
    return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status launch_bwd(const BwdArgs &a)
{
    switch (a.D) {
    case 64: return launch_bwd_d<64>(a);
    case 128: return launch_bwd_d<128>(a);
    case 256: return launch_bwd_d<256>(a);
    default: return FA2_ERR_UNSUPPORTED;
    }
}

}  // namespace fa2
