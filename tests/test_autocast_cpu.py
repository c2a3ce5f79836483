"""fp8_autocast on the host: when the scale update runs ("FP8 低精度训练：
Transformer Engine 简析" §三.3: at autocast exit, for the next step)."""
import pytest


class _FakeState:
    def __init__(self):
        self.calls = []

    def update(self, step, stream=None):
        self.calls.append(step)


def test_update_once_per_exit_with_counting_steps():
    from fp8_delayed_scaling_gb300.autocast import active, fp8_autocast
    st = _FakeState()
    assert active() is None
    for _ in range(3):
        with fp8_autocast(st) as ac:
            assert active() is ac
    assert st.calls == [0, 1, 2] and active() is None
    with fp8_autocast(st, step=10):
        pass
    with fp8_autocast(st):
        pass
    assert st.calls == [0, 1, 2, 10, 11]


def test_no_update_when_disabled_or_the_block_raises():
    from fp8_delayed_scaling_gb300.autocast import active, fp8_autocast
    st = _FakeState()
    with fp8_autocast(st, enabled=False):
        pass
    with pytest.raises(ValueError):
        with fp8_autocast(st):
            raise ValueError("step failed")
    assert st.calls == [] and active() is None
    with fp8_autocast(st):
        with fp8_autocast(st, enabled=False) as inner:
            assert active() is inner
    assert st.calls == [0]
