// Host-side check of the decode kernel's shared-memory carve-up for every
// instantiated (D, G, cache type): regions that take 16-byte accesses start
// on 16-byte boundaries, the stage ring on a 1024-byte boundary (the 128-byte
// swizzle's period), the barriers on 8 bytes, and every warp's merge rows on 8
// bytes (float2 stores).  Built and run by tests/test_layout.py; no GPU.
#include "decode_kernel.cuh"

#include <cstdio>

using namespace pkv::kern;

template <int D, int G, int KV>
int check()
{
    using C = Cfg<D, G, KV>;
    int bad = 0;
    for (int nst = 2; nst <= MAX_STAGES; ++nst)
        for (int batch : {1, 2, 3, 7, 64, 4096})
            for (bool prefix : {false, true}) {
                const Layout L = make_layout<D, G, KV>(nst, batch, prefix);
                const int sixteen[] = {L.stages, L.scales, L.qring, L.merge, L.ps, L.pre, L.lens};
                for (int o : sixteen)
                    bad += o % 16 != 0;
                bad += L.stages % 1024 != 0;
                bad += C::SWIZZLE_OK && C::STAGE_BYTES % 1024 != 0;
                bad += L.bars % 8 != 0 || L.misc % 4 != 0;
                bad += (L.merge / 4) % 2 != 0 || (G * (D + 2)) % 2 != 0;
                bad += L.total > 232448 && nst == 2 && batch <= 64;
            }
    if (bad)
        std::printf("D=%d G=%d KV=%d: %d bad layouts\n", D, G, KV, bad);
    return bad;
}

template <int D, int KV>
int check_groups()
{
    return check<D, 1, KV>() + check<D, 2, KV>() + check<D, 4, KV>() + check<D, 8, KV>();
}

int main()
{
    const int bad = check_groups<64, PKV_F32>() + check_groups<128, PKV_F32>() +
                    check_groups<64, PKV_F16>() + check_groups<128, PKV_F16>() +
                    check_groups<64, PKV_BF16>() + check_groups<128, PKV_BF16>() +
                    check_groups<64, PKV_I8>() + check_groups<128, PKV_I8>() +
                    check_groups<128, PKV_I4>();
    std::printf("layout check: %d bad\n", bad);
    return bad != 0;
}
