"""Save and resume (mt_save / mt_load).

Between steps the GPU holds no model state, so a run saved after step s and
loaded into a fresh model of the same shape (initialised with another seed)
continues bit for bit like the run that never stopped: the kernels and the
host Adam are deterministic for the same inputs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import configs, inputs  # noqa: E402


@pytest.mark.parametrize("name,rt", [("tiny", {}), ("tiny_moe", dict(ckpt_interval=2, pin_store=1))])
def test_save_load_resumes_bit_exact(tmp_path, name, rt):
    c = configs.get(name)
    path = str(tmp_path / "store.bin")
    a = mt.Model(c, seed=7, **rt)
    for s in range(2):
        a.set_tokens(inputs.tokens_for(c, s))
        a.train_step(s)
    a.save(path)
    b = mt.Model(c, seed=99, **rt)  # other initial weights, overwritten by the load
    b.load(path)
    with pytest.raises(mt.MtError) as ei:
        b.train_step(3)  # the resumed run continues at step 2
    assert ei.value.status == -2
    losses = []
    for m in (a, b):
        m.set_tokens(inputs.tokens_for(c, 2))
        losses.append(m.train_step(2))
        m.sync()
    assert losses[0] == losses[1]
    for j in range(c["n_layers"] + 2):
        for region in (mt.REGION_W, mt.REGION_G, mt.REGION_MASTER, mt.REGION_M, mt.REGION_V):
            x, y = a.read(j, region), b.read(j, region)
            bad = np.flatnonzero(x.view(np.uint8) != y.view(np.uint8)) // x.itemsize
            where = [t for t, (off, r, cc) in enumerate(a.layout[j]["tensors"]) if bad.size and off <= bad[0] < off + r * cc]
            assert bad.size == 0, (j, region, bad.size, bad[:8], where, x[bad[:4]], y[bad[:4]])
    a.close()
    b.close()


def test_load_rejects_another_shape(tmp_path):
    c = configs.get("tiny")
    path = str(tmp_path / "store.bin")
    a = mt.Model(c, seed=7)
    a.save(path)
    a.close()
    d = mt.Model(configs.get("tiny", n_layers=3))
    with pytest.raises(mt.MtError) as ei:
        d.load(path)
    assert ei.value.status == -1
    with pytest.raises(mt.MtError) as ei:
        d.load(str(tmp_path / "missing.bin"))
    assert ei.value.status == -1
    d.set_tokens(inputs.tokens_for(configs.get("tiny", n_layers=3), 0))
    assert np.isfinite(d.train_step(0))  # refused loads leave the model usable
    d.close()
