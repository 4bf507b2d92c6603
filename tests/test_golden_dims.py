"""The dimensions the pages print (tests/golden/model_dims.txt) against the
oracle's constants and the synthetic workloads' shapes."""
import os

import gdn_inputs
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _load():
    rows, scal = {}, {}
    for line in open(os.path.join(HERE, "golden", "model_dims.txt")):
        line = line.split("#")[0].split()
        if len(line) == 5:
            rows[line[0]] = tuple(int(v) for v in line[1:])
        elif len(line) == 2:
            scal[line[0]] = float(line[1])
    return rows, scal


def test_printed_dims():
    rows, scal = _load()
    assert oracle.D == 128 and oracle.KW == int(scal["conv_kernel"]) and oracle.EPS == scal["eps"]
    for model, (hk, hv, d, inner) in rows.items():
        assert d == oracle.D and hv * d == inner, model
    # the workloads use exactly these head counts; fused width 128*(2*H_k+H_v)
    assert rows["27B"][:2] == (16, 48) and rows["35B-A3B"][:2] == (16, 32)
    c = gdn_inputs.make_case("t", Hk=16, Hv=48, lengths=[1])
    assert c.C == 10240 and c.z.shape[1] == rows["27B"][3]
    c = gdn_inputs.make_case("t", Hk=16, Hv=32, B=1)
    assert c.C == 8192 and c.z.shape[1] == rows["35B-A3B"][3]
