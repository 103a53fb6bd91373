"""Random problems (seeded) through the C ABI against the oracle: dtypes
(f16, bf16, e4m3 with scales), group sizes, query blocks, contiguous and
paged caches (pages of 8, 16 and 64 tokens, shuffled tables), planned and
forced split counts, output dtypes, lse on or off, the CUDA-core consumer
where it applies, and lengths from 0 to the capacity.  Canary guards check
that nothing is written outside out, lse and the workspace."""
import numpy as np
import pytest
import torch

import fd_inputs
import split_kv_gb300 as fd
from gpu_util import assert_parity, oracle_all, run_decode

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
FP8 = hasattr(torch, "float8_e4m3fn")
N_CASES = 120


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)
    fd.fd_device_status(clear=True)
    yield


def _case(i):
    rng = np.random.default_rng(5000 + i)
    kv = str(rng.choice(["f16", "bf16", "e4m3"] if FP8 else ["f16", "bf16"]))
    qd = kv if kv != "e4m3" else str(rng.choice(["f16", "bf16"]))
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    ql = int(rng.choice([1, 1, 1, 2, 3, 4, 8]))
    while G * ql > 64:
        ql = max(1, ql // 2)
    Hkv = int(rng.integers(1, 4))
    B = int(rng.integers(1, 5))
    ps = int(rng.choice([0, 0, 8, 16, 64]))
    T = int(rng.integers(1, 40000 if rng.random() < 0.1 else 3000))
    lens = rng.integers(0, T + 1, size=B)
    lens[rng.integers(0, B)] = T                     # one sequence at the capacity
    if B > 1 and rng.random() < 0.5:
        lens[rng.integers(0, B)] = 0                 # an empty one
    S = int(rng.choice([0, 0, 1, int(rng.integers(2, 129))]))
    out_dtype = [torch.float32, torch.float16, torch.bfloat16][int(rng.integers(0, 3))]
    cuda_cores = kv != "e4m3" and ql == 1 and G in (1, 2, 4, 8) and rng.random() < 0.3
    return dict(kv=kv, qd=qd, G=G, ql=ql, Hkv=Hkv, B=B, ps=ps, T=T, lens=lens.astype(np.int32),
                S=S, out_dtype=out_dtype, cuda_cores=cuda_cores, seed=6000 + 10 * i)


N_WIDE = 32


def _wide_case(i):
    """A query block of 17-256 columns per KV head: the tcgen05 kernels
    (17-64, 65-128 on a 16-bit cache) and column blocks (fp8, or more than
    128 columns); a third of the cases in each column range."""
    rng = np.random.default_rng(7000 + i)
    c = _case(10_000 + i)
    lo, hi = [(17, 64), (65, 128), (129, 256)][i % 3]
    while True:
        G = int(rng.choice([3, 4, 5, 6, 8, 12, 16]))
        ql = int(rng.choice([2, 3, 4, 5, 8, 12, 16]))
        if lo <= G * ql <= hi:
            break
    if rng.random() < 0.8:                               # mostly 16-bit caches
        c["kv"] = c["qd"] = str(rng.choice(["f16", "bf16"]))
    T = int(rng.integers(1, 2500))
    B = int(rng.integers(1, 4))
    lens = rng.integers(0, T + 1, size=B)
    lens[rng.integers(0, B)] = T
    c.update(G=G, ql=ql, Hkv=int(rng.integers(1, 3)), B=B, T=T, lens=lens.astype(np.int32),
             cuda_cores=False, seed=8000 + 10 * i)
    return c


def _run_case(c, what_prefix):
    B, G, ql, Hkv, T, ps, D = c["B"], c["G"], c["ql"], c["Hkv"], c["T"], c["ps"], 128
    B, G, ql, Hkv, T, ps, D = c["B"], c["G"], c["ql"], c["Hkv"], c["T"], c["ps"], 128
    Hq = G * Hkv
    seed = c["seed"]
    q = fd_inputs.randn((B, ql, Hq, D) if ql > 1 else (B, Hq, D), c["qd"], seed, device=DEV)
    sc, okw = {}, {}
    if ps:
        mp = -(-T // ps)
        n_pages = B * mp + 3
        shape = (n_pages, Hkv, ps, D)
    else:
        shape = (B, Hkv, T, D)
    if c["kv"] == "e4m3":
        k = fd_inputs.randn_fp8(shape, seed + 1, device=DEV, gain=16.0)
        v = fd_inputs.randn_fp8(shape, seed + 2, device=DEV, gain=16.0)
        sc = dict(k_scale=1 / 16, v_scale=1 / 16)
        okw = dict(kv_dtype="e4m3", **sc)
    else:
        k = fd_inputs.randn(shape, c["kv"], seed + 1, device=DEV)
        v = fd_inputs.randn(shape, c["kv"], seed + 2, device=DEV)
    bt = None
    if ps:
        bt = fd_inputs.page_permutation(seed + 3, n_pages)[:B * mp].reshape(B, mp).copy()
        okw.update(page_size=ps, block_table=bt)
    flags = fd.FD_FLAG_CUDA_CORES if c["cuda_cores"] else 0
    got_o, got_l, S = run_decode(q, k, v, c["lens"], page_size=ps, block_table=bt, n_splits=c["S"],
                                 out_dtype=c["out_dtype"], flags=flags, **sc)
    ref_o, ref_l = oracle_all(q, k, v, c["lens"], c["qd"], Hkv, **okw)
    if c["out_dtype"] != torch.float32:
        # the output is rounded to 16 bits: compare with the rounded reference
        ref_o = torch.from_numpy(ref_o).to(c["out_dtype"]).double().numpy()
    what = (f"{what_prefix}: kv={c['kv']} q={c['qd']} G={G} q_len={ql} Hkv={Hkv} B={B} page={ps} "
            f"T={T} lens={c['lens'].tolist()} S={S} out={c['out_dtype']} cuda_cores={c['cuda_cores']}")
    assert_parity(got_o, got_l, ref_o, ref_l, what)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_problem(i):
    _run_case(_case(i), f"case {i}")


@pytest.mark.parametrize("i", range(N_WIDE))
def test_random_wide_query_block(i):
    _run_case(_wide_case(i), f"wide case {i}")
