"""Host-only checks of the window-vote planner through snapkv_vote_plan (no GPU needed):
the plans the measured workloads run with, and on a seeded sweep of shapes and SM counts
the limits every plan must respect -- a single-pass plan holds two jobs' key tiles per CTA
in tensor memory (512 columns of the job's query rows) and, with an exchange, streams at
least 4 tiles per CTA and job; a two-pass plan gives each CTA at least one key tile of
every job; the exchange records cover g partial statistics per row and an arrival
counter per job."""

import math

import numpy as np
import pytest

import attention_score_kv_snapkv_gb300 as kvc

TILE = 128


def key_tiles(L, R, Wq, rt):
    """Key tiles a row tile sees: its rows are window rows r0.. of the G query heads, and
    row r sees the keys up to position L - Wq + r (causal inside the window)."""
    nrows = min(TILE, R - rt * TILE)
    r0 = (rt * TILE) % Wq
    last = Wq - 1 if r0 + nrows > Wq else r0 + nrows - 1
    return math.ceil((L - Wq + last + 1) / TILE)


def align256(n):
    return (n + 255) // 256 * 256


def test_plans_of_the_measured_workloads():
    # Mistral-7B-shaped compression: 128 window rows per unit -> two passes, groups of 8
    p = kvc.snapkv_vote_plan(32, 2, 32, 8, 128, 16384, 32, 32, 7, 1024, num_sms=152)
    assert (p["single"], p["g"], p["groups"], p["row_tiles"], p["rows_per_tile"]) == (0, 8, 19, 1, 128)
    # long context: 32 rows per unit -> one pass, 147 CTAs per job (7 tiles of 1024 each)
    p = kvc.snapkv_vote_plan(8, 1, 32, 32, 128, 131072, 32, 32, 7, 1024, num_sms=152)
    assert (p["single"], p["g"], p["groups"], p["row_tiles"], p["rows_per_tile"]) == (1, 147, 1, 1, 32)
    # H2O prefill scores (every prompt row votes): two passes, one CTA per job
    p = kvc.snapkv_vote_plan(1, 64, 32, 32, 128, 2048, 2048, 204, 1, 408, 409, num_sms=152)
    assert (p["single"], p["g"], p["row_tiles"], p["exchange_bytes"]) == (0, 1, 16, 0)


def draw(seed):
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.randint(1, 9))
    G = int(r.randint(1, 9))
    L = max(1, int(np.exp(r.uniform(0.0, np.log(300000.0)))))
    Wq = L if r.rand() < 0.15 else int(r.randint(1, min(L, 160) + 1))
    Ly, B = int(r.randint(1, 33)), int(r.randint(1, 5))
    sms = int(r.choice([152, 148, 132, 76, 16]))
    return Ly, B, G * Hkv, Hkv, D, L, Wq, sms


def draw_few_rows(seed):
    """Long prompts with at most 64 voting rows per unit: the single-pass kernel's shapes."""
    r = np.random.RandomState(seed)
    D = int(r.choice([64, 128]))
    Hkv = int(r.randint(1, 9))
    G = int(r.randint(1, 5))
    L = int(np.exp(r.uniform(np.log(2048.0), np.log(300000.0))))
    Wq = int(r.randint(1, 64 // G + 1))
    Ly, B = int(r.randint(1, 9)), int(r.randint(1, 3))
    sms = int(r.choice([152, 148, 132, 76]))
    return Ly, B, G * Hkv, Hkv, D, L, Wq, sms


@pytest.mark.parametrize("seed", list(range(60)) + list(range(1000, 1030)))
def test_plan_respects_its_limits(seed):
    Ly, B, Hq, Hkv, D, L, Wq, sms = draw(seed) if seed < 1000 else draw_few_rows(seed)
    G = Hq // Hkv
    R = G * Wq
    units = Ly * B * Hkv
    if units * L > 2 ** 31 - 1 or units * R > 2 ** 31 - 1:
        pytest.skip("beyond the row limit")
    p = kvc.snapkv_vote_plan(Ly, B, Hq, Hkv, D, L, Wq, Wq, 1, L, num_sms=sms)
    row_tiles = math.ceil(R / TILE)
    nkt = [key_tiles(L, R, Wq, rt) for rt in range(row_tiles)]
    g = p["g"]
    jobs = units * row_tiles
    assert p["row_tiles"] == row_tiles
    assert 1 <= g <= sms and p["groups"] == sms // g
    if p["single"]:
        qr = TILE if R >= TILE else (R + 15) // 16 * 16
        assert p["rows_per_tile"] == qr
        tpc = math.ceil(max(nkt) / g)
        assert 2 * tpc <= 512 // qr           # two jobs of tiles fit tensor memory
        if g > 1:
            assert tpc >= 4                   # enough streaming to cover an exchange
    else:
        qr = TILE
        assert p["rows_per_tile"] == TILE
        assert g <= min(nkt)                  # every CTA of a group has a tile of each job
    expect = align256(jobs * g * qr * 8 + jobs * 4) if g > 1 else 0
    assert p["exchange_bytes"] == expect


def test_rejected_sizes_raise_with_the_call_codes():
    with pytest.raises(kvc.KVCError) as e:       # Hq not a multiple of Hkv
        kvc.snapkv_vote_plan(1, 1, 3, 2, 128, 100, 8, 8, 7, 64, num_sms=152)
    assert e.value.code == 2
    with pytest.raises(kvc.KVCError) as e:       # more window queries than prompt positions
        kvc.snapkv_vote_plan(1, 1, 4, 4, 64, 10, 12, 8, 7, 9, num_sms=152)
    assert e.value.code == 2
    with pytest.raises(kvc.KVCError) as e:       # even pool kernel
        kvc.snapkv_vote_plan(1, 1, 4, 4, 64, 100, 8, 8, 4, 16, num_sms=152)
    assert e.value.code == 2
    with pytest.raises(kvc.KVCError) as e:       # budget below the kept window
        kvc.snapkv_vote_plan(1, 1, 4, 4, 64, 100, 8, 16, 7, 12, num_sms=152)
    assert e.value.code == 4


def test_h2o_step_plans_on_the_host():
    """h2o_step_ctas_per_unit is host arithmetic too (160 SMs assumed without a device):
    one CTA per unit for the OPT-6.7B-shaped step, the split step when a unit's logits do
    not fit one CTA's shared memory, 0 for sizes the step rejects."""
    assert kvc.h2o_step_ctas_per_unit(32, 64, 32, 32, 128, 204, 204) == 1
    assert kvc.h2o_step_ctas_per_unit(8, 1, 32, 32, 128, 13107, 13107) > 1
    assert kvc.h2o_step_ctas_per_unit(1, 1, 36, 4, 128, 8, 8) == 0      # 9 query heads per KV head
    assert kvc.h2o_step_ctas_per_unit(1, 1, 4, 4, 128, 8, 0) == 0       # no recent window
    assert kvc.h2o_step_ctas_per_unit(1, 1, 4, 4, 96, 8, 8) == 0        # head dim 96


def test_readme_example_calls_existing_entry_points():
    import os
    import re
    from conftest import ROOT
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks
    names = set(re.findall(r"kvc\.([a-z_0-9]+)\(", "".join(blocks)))
    assert names
    for n in sorted(names):
        assert callable(getattr(kvc, n, None)), n
