"""The tiled weight layout written by q4_tile, byte for byte against a plain
host description of the format, on shapes with a ragged last row tile, a
partial last column chunk, the gate/up pairing and expert stacks.

Format (include/verify.h, q4_tile): per (128-row tile, chunk of G 64-column
groups; G = 4 for dense products, 2 for the experts' gate/up and down
matrices) one block = scales [128 rows][G groups] bf16, biases likewise,
then for each group present: for 16-row block b and lane L = 4g + c the words
(row 16b+g W0, row 16b+g+8 W0, row 16b+g W1, row 16b+g+8 W1), where Ww holds
columns 16c + 8w .. 16c + 8w + 7 of the group with nibble p taken from
column 16c + 8w + sigma(p), sigma = (0 4 2 6 1 5 3 7).  Rows past the matrix
are zero.  With the gate/up pairing tile t = gate rows 64t.., then up rows
I + 64t.. .
"""
import numpy as np
import pytest

from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu

SIGMA = [0, 4, 2, 6, 1, 5, 3, 7]


def permute_word(u):
    out = 0
    for p in range(8):
        out |= ((int(u) >> (4 * SIGMA[p])) & 0xF) << (4 * p)
    return out


def tile_host(packed, scales, biases, N, K, gate_up, GR=4):
    """Tiled bytes of one matrix [N, K] (row layout: packed uint32 [N, K/8],
    scales/biases uint16 [N, K/64]), GR groups per chunk."""
    KG, KC, KW = K // 64, (K // 64 + GR - 1) // GR, K // 8
    RT = N // 128 if gate_up else (N + 127) // 128
    out = bytearray()
    for rt in range(RT):
        if gate_up:
            rows = [64 * rt + i for i in range(64)] + [N // 2 + 64 * rt + i for i in range(64)]
        else:
            rows = [rt * 128 + i if rt * 128 + i < N else -1 for i in range(128)]
        for kc in range(KC):
            gcount = min(GR, KG - GR * kc)
            sb = np.zeros((2, 128, GR), np.uint16)
            for i, r in enumerate(rows):
                if r >= 0:
                    for G in range(gcount):
                        sb[0, i, G] = scales[r, GR * kc + G]
                        sb[1, i, G] = biases[r, GR * kc + G]
            out += sb.tobytes()
            for G in range(gcount):
                blk = np.zeros((8, 32, 4), np.uint32)
                for b in range(8):
                    for lane in range(32):
                        g, c = lane >> 2, lane & 3
                        r0, r1 = rows[16 * b + g], rows[16 * b + g + 8]
                        wi = 8 * (GR * kc + G) + 2 * c
                        w = lambda r, o: permute_word(packed[r, wi + o]) if r >= 0 else 0  # noqa: E731
                        blk[b, lane] = [w(r0, 0), w(r1, 0), w(r0, 1), w(r1, 1)]
                out += blk.tobytes()
    return bytes(out)


@pytest.fixture(scope="module")
def vf():
    v = B.Verify(0)
    yield v
    v.close()


@pytest.mark.parametrize("N,K,E,kind", [(200, 576, 1, B.TILE_DENSE), (128, 256, 1, B.TILE_DENSE),
                                        (384, 192, 2, B.TILE_GATE_UP), (130, 640, 2, B.TILE_DENSE),
                                        (256, 448, 3, B.TILE_GATE_UP), (130, 640, 2, B.TILE_DOWN),
                                        (200, 576, 1, B.TILE_DOWN), (384, 64, 1, B.TILE_DOWN)])
def test_tiled_bytes_match_the_format(vf, N, K, E, kind):
    import torch

    m = S.q4_matrix(7, f"tile.{N}.{K}", N, K, n_experts=E if E > 1 else None)
    keep = (dev(m.packed), dev(m.scales), dev(m.biases))  # alive while the struct points at them
    W = B.q4_experts(*keep) if E > 1 else B.q4_weight(*keep)
    gate_up = kind == B.TILE_GATE_UP
    t = vf.tile(W, gate_up=gate_up, down=kind == B.TILE_DOWN)
    torch.cuda.synchronize()
    got = host(t.buf).tobytes()
    P = m.packed.reshape(E, N, K // 8)
    Sc = m.scales.reshape(E, N, K // 64)
    Bi = m.biases.reshape(E, N, K // 64)
    GR = 4 if kind == B.TILE_DENSE else 2
    want = b"".join(tile_host(P[e], Sc[e], Bi[e], N, K, gate_up, GR) for e in range(E))
    assert len(got) == len(want) == vf.lib.q4_tiled_bytes(N, K, E, kind)
    assert got == want
    s = t.struct.w if E > 1 else t.struct
    layout = {B.TILE_DENSE: B.TILED, B.TILE_GATE_UP: B.TILED_GATE_UP, B.TILE_DOWN: B.TILED_DOWN}[kind]
    assert s.layout == layout and not s.scales and not s.biases
    del keep


def test_tile_rejects_bad_arguments(vf):
    import torch

    m = S.q4_matrix(7, "tile.err", 128, 256)
    keep = (dev(m.packed), dev(m.scales), dev(m.biases))
    W = B.q4_weight(*keep)
    part = (keep[0][:96], keep[1][:96], keep[2][:96])
    with pytest.raises(B.VerifyError) as e:  # gate/up pairing needs 2I with I % 64 == 0
        vf.tile(B.q4_weight(*part), gate_up=True)
    assert e.value.status == B.EUNSUPPORTED
    t = vf.tile(W)
    with pytest.raises(B.VerifyError) as e:  # a tiled matrix is not a q4_tile input
        vf.tile(t.struct)
    assert e.value.status == B.EINVAL
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = B.Q4Weight()
    import ctypes as C
    st = vf.lib.q4_tile(vf.ctx, C.byref(W), 1, 0, C.c_void_p(small.data_ptr()), 16, C.byref(out), None)
    assert st == B.EINVAL  # dst smaller than q4_tiled_bytes
    assert vf.lib.q4_tiled_bytes(128, 100, 1, 0) == -1
    assert vf.lib.q4_tiled_bytes(128, 256, 1, 3) == -1  # no such tile kind
    with pytest.raises(B.VerifyError) as e:  # the experts' down layout is not a dense operand
        vf.q4_qmv_k(vf.tile(W, down=True).struct, torch.zeros((1, 256), dtype=torch.int16, device="cuda"), 1,
                    torch.zeros((1, 128), device="cuda"))
    assert e.value.status == B.EINVAL
