"""Bias checkpoint (host only): bit-exact round trip, refused bad files."""
import numpy as np
import pytest

from mixture_experts_layer_gemms_b300.checkpoint import load_bias, save_bias


def test_round_trip_bit_exact(tmp_path):
    b = np.array([0.0, -0.0, 1e-3, -2.5e-7, 3.4e38, np.float32(1) / 3],
                 dtype=np.float32)
    p = str(tmp_path / "b.ckpt")
    save_bias(p, b, 17)
    got, step = load_bias(p)
    assert step == 17
    assert got.tobytes() == b.tobytes()


def test_refuses_bad_files(tmp_path):
    p = tmp_path / "x.ckpt"
    p.write_bytes(b"NOTABIAS" + b"\0" * 12)
    with pytest.raises(ValueError):
        load_bias(str(p))
    save_bias(str(p), np.zeros(8, np.float32), 0)
    raw = p.read_bytes()
    p.write_bytes(raw[:-4])
    with pytest.raises(ValueError):
        load_bias(str(p))
    with pytest.raises(ValueError):
        save_bias(str(p), np.zeros(8, np.float64), 0)
