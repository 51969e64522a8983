"""GPU parity on model shapes the workloads do not use: widths that are
multiples of 16 but not of 32, 64 or 128 (the CUDA-core and direct GEMV paths
take every ragged K tail, the tensor path steps aside where K is not a
multiple of 128, and the prefill GEMMs pad K to their 32-wide chunks), and a
GQA group of 1 (as many kv heads as q heads). Frames teacher-forced with
sampling on, and a prompt pass, against the oracle."""
import numpy as np
import pytest

from codebook_decode_gb300 import configs, synth
from codebook_decode_gb300.engine import to_dev_u16
from gpu_helpers import TOL_BF16, ParityRun, free

pytestmark = pytest.mark.gpu

ODD = configs.Dims(**{**configs.TINY.as_dict(), "hidden": 528, "ffn": 1552, "cp_hidden": 272, "cp_ffn": 784})
GQA1 = configs.Dims(**{**configs.TINY.as_dict(), "n_kv_heads": 8, "cp_n_kv_heads": 4})


def sessions(d, B, prefixes, frames):
    return synth.Sessions(d, B, prefixes[:B], [0] * B, frames, 2300 + B, temperature=0.9, top_k=50,
                          rep_penalty=1.05)


@pytest.mark.parametrize("dims", [ODD, GQA1], ids=["odd_widths", "gqa_group_1"])
@pytest.mark.parametrize("B", [3, 9])
def test_frames_match_oracle(dims, B):
    w = synth.make_weights(dims, 1100)
    s = sessions(dims, B, [5, 33, 17, 2, 40, 11, 25, 8, 30], 3)
    run = ParityRun(dims, w, s, 3, shuffle=True).run()
    try:
        assert run.max_rel() < TOL_BF16, run.max_rel()
        assert run.confident_agree == run.confident
        run.check_state()
        run.check_kv()
    finally:
        free(run)


@pytest.mark.parametrize("dims", [ODD, GQA1], ids=["odd_widths", "gqa_group_1"])
@pytest.mark.parametrize("n_tok", [37, 320])
def test_prefill_matches_oracle(dims, n_tok):
    """2 x 320 rows: one K-slice per gate/up tile, SwiGLU in its epilogue."""
    w = synth.make_weights(dims, 1101)
    s = sessions(dims, 2, [9, 30], n_tok + 3)
    run = ParityRun(dims, w, s, n_tok + 2, shuffle=True)
    try:
        e = s.prompt_embeds(n_tok)
        run.eng.prefill(to_dev_u16(e, run.eng.dev))
        assert run.eng.status() == (0, 0)
        run.O.talker_prefill(run.rows, run.kv, run.cap, e)
        run.check_state()
        run.check_kv()
        run.run(frames=1)
        assert run.max_rel() < TOL_BF16, run.max_rel()
    finally:
        free(run)
