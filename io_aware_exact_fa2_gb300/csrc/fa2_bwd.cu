// fa2_bwd.cu -- host-side launch of the backward pass ("Chapter 08: Flash
// Attention -- blocked attention", section 6): the Delta kernel, then dQ (query
// tiles resident), then dK and dV (key/value tiles resident), all on one stream.
#include <atomic>

#include "fa2_bwd_kernel.cuh"
#include "fa2_launch.cuh"

namespace fa2 {

// dK/dV: 128 keys resident, query tiles of 64 streamed through a 4-stage ring
// (dV, dK and two 64-column score pairs fill TMEM; K and V stay in shared memory);
// dQ: 128 queries resident, key tiles of 64 through a 4-stage ring.  Two score
// buffer pairs let one step's MMAs run while the previous step's elementwise
// work finishes.
template <int D>
using BwdKV = BwdCfg<D, 128, 64, 4, 8>;
template <int D>
using BwdQ = BwdCfg<D, 128, 64, 4, 8>;
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

template <int D>
static fa2_status launch_bwd_d(const BwdArgs &a)
{
    using CKV = BwdKV<D>;
    using CQ = BwdQ<D>;
    const int BH = a.B * a.H;
    CUtensorMap q_res, do_res, k_str, v_str, k_res, v_res, q_str, do_str;
    if (!encode_bhld(a.encode, &q_res, a.q, D, a.Lq, BH, CQ::RES) ||
        !encode_bhld(a.encode, &do_res, a.dout, D, a.Lq, BH, CQ::RES) ||
        !encode_bhld(a.encode, &k_str, a.k, D, a.Lk, BH, CQ::STR) ||
        !encode_bhld(a.encode, &v_str, a.v, D, a.Lk, BH, CQ::STR) ||
        !encode_bhld(a.encode, &k_res, a.k, D, a.Lk, BH, CKV::RES) ||
        !encode_bhld(a.encode, &v_res, a.v, D, a.Lk, BH, CKV::RES) ||
        !encode_bhld(a.encode, &q_str, a.q, D, a.Lq, BH, CKV::STR) ||
        !encode_bhld(a.encode, &do_str, a.dout, D, a.Lq, BH, CKV::STR))
        return FA2_ERR_CUDA;
    BwdParams p;
    const int n_stat_tiles = (a.Lq + BWD_STAT_ROWS - 1) / BWD_STAT_ROWS;
    p.stats = a.stats;
    p.n_stat_tiles = n_stat_tiles;
    p.dq = static_cast<uint16_t *>(a.dq);
    p.dk = static_cast<uint16_t *>(a.dk);
    p.dv = static_cast<uint16_t *>(a.dv);
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
            n_stat_tiles, rows);
        const long long n_qt = (a.Lq + CQ::RES - 1) / CQ::RES;
        fa2_bwd_q_kernel<CQ><<<static_cast<unsigned>(n_qt * BH), CQ::NUM_THREADS, CQ::SMEM_BYTES, a.stream>>>(
            q_res, do_res, k_str, v_str, p);
    }
    const long long n_kt = (a.Lk + CKV::RES - 1) / CKV::RES;
    fa2_bwd_kv_kernel<CKV><<<static_cast<unsigned>(n_kt * BH), CKV::NUM_THREADS, CKV::SMEM_BYTES, a.stream>>>(
        k_res, v_res, q_str, do_str, p);
    return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

fa2_status launch_bwd(const BwdArgs &a)
{
    switch (a.D) {
    case 64: return launch_bwd_d<64>(a);
    case 128: return launch_bwd_d<128>(a);
    default: return FA2_ERR_UNSUPPORTED;
    }
}

}  // namespace fa2
