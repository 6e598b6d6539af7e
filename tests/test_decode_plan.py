"""Host logic of the decode launch's work division (qrr_plan_decode_units):
every stage of every tile is taken exactly once, the LoRA stage last, the
pieces of a split tile are numbered and counted consistently, and the
stream-K cut gives every CTA the same number of stages to within one.  No GPU
is needed: the query runs the library's own planning on the host."""

import pytest

from quantized_rl_rollout_gb300 import configs, qrr

LAYERS_8B = [(l.n, l.k, 32) for l in configs.LAYERS_8B]
LAYERS_32B = [(5120, 5120, 64), (1024, 5120, 64), (1024, 5120, 64), (5120, 5120, 64), (27648, 5120, 64),
              (27648, 5120, 64), (5120, 27648, 64)]
MIXED = [(384, 1024, 32), (128, 256, 8), (256, 2048, 0), (512, 768, 64)]


def _m_tiles(m):
    bn = 16 if m <= 16 else 32 if m <= 32 else 64
    return (m + bn - 1) // bn


def _check_cover(m, shapes, units):
    """Every tile's K stages once, its LoRA stage (r > 0) once and last."""
    mt_n = _m_tiles(m)
    seen = {}
    for u in units:
        key = (u["layer"], u["m_tile"], u["n_tile"])
        seen.setdefault(key, []).append(u)
    expected = {(j, mt, nt) for j, (n, k, r) in enumerate(shapes) for mt in range(mt_n) for nt in range(n // 128)}
    assert set(seen) == expected
    for (j, mt, nt), pieces in seen.items():
        n, k, r = shapes[j]
        kc = k // 256
        counts = {p["pieces"] for p in pieces}
        assert counts == {len(pieces)}, (j, mt, nt, counts, len(pieces))
        assert sorted(p["piece"] for p in pieces) == list(range(len(pieces)))
        covered = []
        for p in pieces:
            covered.extend(range(p["c0"], p["c0"] + p["nk"]))
        assert sorted(covered) == list(range(kc)), (j, mt, nt)
        loras = [p for p in pieces if p["lora"]]
        if r > 0:
            assert len(loras) == 1 and loras[0]["piece"] == len(pieces) - 1
        else:
            assert not loras


def _cta_stages(units, offsets):
    return [sum(u["nk"] + u["lora"] for u in units[offsets[b]:offsets[b + 1]]) for b in range(len(offsets) - 1)]


@pytest.mark.parametrize("m", [1, 8, 16, 32])
@pytest.mark.parametrize("grid", [152, 148, 7, 1])
@pytest.mark.parametrize("shapes", [LAYERS_8B, MIXED, LAYERS_32B], ids=["8b", "mixed", "32b"])
def test_stream_k_cut(m, grid, shapes):
    units, offsets = qrr.plan_decode_units(m, shapes, grid)
    _check_cover(m, shapes, units)
    total = sum((n // 128) * _m_tiles(m) * (k // 256 + (1 if r else 0)) for n, k, r in shapes)
    used = len(offsets) - 1
    assert used == min(grid, total)
    assert offsets[0] == 0 and offsets[-1] == len(units)
    assert all(a <= b for a, b in zip(offsets, offsets[1:]))
    per = _cta_stages(units, offsets)
    assert sum(per) == total
    assert max(per) - min(per) <= 1
    # a split tile's pieces run in piece order over the CTAs
    where = {}
    for b in range(used):
        for u in units[offsets[b]:offsets[b + 1]]:
            where[(u["layer"], u["m_tile"], u["n_tile"], u["piece"])] = b
    for (j, mt, nt, p), b in where.items():
        if p > 0:
            assert where[(j, mt, nt, p - 1)] <= b


@pytest.mark.parametrize("m", [33, 48, 64])
@pytest.mark.parametrize("grid", [152, 20])
@pytest.mark.parametrize("shapes", [LAYERS_8B, MIXED], ids=["8b", "mixed"])
def test_split_k_longest_first(m, grid, shapes):
    units, offsets = qrr.plan_decode_units(m, shapes, grid)
    _check_cover(m, shapes, units)
    # at most one unit of difference between the most and least loaded CTA,
    # in stages plus the epilogue allowance the planner uses
    def cost(u):
        return u["nk"] + u["lora"] + (3.0 if u["pieces"] > 1 else 0.5)
    loads = [sum(cost(u) for u in units[offsets[b]:offsets[b + 1]]) for b in range(len(offsets) - 1)]
    assert max(loads) - min(loads) <= max(cost(u) for u in units) + 1e-9


def test_plan_rejects_bad_arguments():
    with pytest.raises(qrr.QrrError):
        qrr.plan_decode_units(65, LAYERS_8B, 152)  # not a decode size
    with pytest.raises(qrr.QrrError):
        qrr.plan_decode_units(1, [(4096, 4000, 32)], 152)  # K % 256
    with pytest.raises(qrr.QrrError):
        qrr.plan_decode_units(1, [(4000, 4096, 32)], 152)  # N % 128
    with pytest.raises(qrr.QrrError):
        qrr.plan_decode_units(1, [(4096, 4096, 12)], 152)  # rank not a multiple of 8
    with pytest.raises(qrr.QrrError):
        qrr.plan_decode_units(1, LAYERS_8B, 0)  # no CTA
    with pytest.raises(qrr.QrrError):
        qrr.plan_decode_units(1, LAYERS_8B, 152, max_units=10)  # table too small
