"""Host-side logic of bench.py without a GPU: the max-over-ranks timing and
barrier across two gloo ranks (the N > 1 replica path), and the reference
arm's JSON line (the CPU oracle)."""
import glob
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_init()
    assert (r, w) == (rank, world)
    bench.barrier()
    m = bench.reduce_max(10.0 + rank)
    q.put((rank, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "cpu_baseline", "e2e", "higher_is_better"):
        assert k in line
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0


def test_gpu_arm_line_has_every_contract_key():
    # The GPU arm only runs on a GPU, so its JSON line is checked statically:
    # the dict literal gpu_arm returns carries every key the bench contract
    # names (nested ones too), and main() adds the CPU baseline at N = 1.
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    fn = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "gpu_arm")
    out = next(n.value for n in ast.walk(fn) if isinstance(n, ast.Assign)
               and any(isinstance(t, ast.Name) and t.id == "out" for t in n.targets)
               and isinstance(n.value, ast.Dict))

    def keys(d):
        return {k.value: v for k, v in zip(d.keys, d.values) if isinstance(k, ast.Constant)}

    top = keys(out)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "clocks", "gpu_launches"):
        assert k in top, k
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(keys(top["roofline"]))
    assert {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(keys(top["e2e"]))
    assert "workload" in keys(top["config"]) and "l2" in keys(top["config"])
    main = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "main")
    assert "cpu_baseline" in ast.unparse(main)


GPU_ONLY_SOURCES = ["bench.py", "__graft_entry__.py", "bit_weight_only_packed_gb300/qmv.py",
                    "synth/__init__.py", "oracle/__init__.py", "tests/gpu_util.py",
                    "tests/test_zz_no_alloc.py"] + sorted(
    os.path.relpath(p, ROOT) for p in glob.glob(os.path.join(ROOT, "tests", "test_gpu_*.py")))


@pytest.mark.parametrize("path", GPU_ONLY_SOURCES)
def test_no_undefined_global_names(path):
    # Much of this code runs only on a GPU; a name read as a global in any
    # function (closures resolved) must be defined at module level or be a
    # builtin, so a typo cannot wait for the GPU run to surface.
    import builtins
    import symtable
    top = symtable.symtable(open(os.path.join(ROOT, path)).read(), path, "exec")
    defined = {s.get_name() for s in top.get_symbols() if s.is_assigned() or s.is_imported()}
    defined |= set(dir(builtins)) | {"__file__", "__name__"}
    bad = []

    def walk(t):
        for s in t.get_symbols():
            if s.is_global() and s.is_referenced() and s.get_name() not in defined:
                bad.append((t.get_name(), s.get_name()))
        for c in t.get_children():
            walk(c)

    walk(top)
    assert not bad, bad
