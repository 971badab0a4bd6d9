"""The guarded-buffer harness of the GPU canary tests, checked on the CPU with fake kernels:
in-bounds writes pass, a write past either end or a skipped element is caught."""
import pytest

from canary import PAD, fully_written, guarded, intact

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_harness_sees_exact_coverage_and_stray_writes(kind):
    flat, view = guarded((2, 3, 5, 7), kind, "cpu")
    assert intact(flat, kind) and not fully_written(view)
    view.fill_(1.0)                                    # a kernel that writes exactly its output
    assert intact(flat, kind) and fully_written(view)
    flat[PAD + view.numel()] = 0.0                     # one element past the end
    assert not intact(flat, kind)
    flat2, view2 = guarded((4, 8), kind, "cpu")
    view2.fill_(2.0)
    flat2[PAD - 1] = 0.0                               # one element before the start
    assert not intact(flat2, kind)
    flat3, view3 = guarded((4, 8), kind, "cpu")
    view3.fill_(3.0)
    view3[3, 7] = float("nan")                         # an element left unwritten
    assert intact(flat3, kind) and not fully_written(view3)


def test_guarded_views_are_contiguous_and_16_byte_aligned_inside_the_buffer():
    flat, view = guarded((3, 100), "bf16", "cpu")
    assert view.is_contiguous() and (view.data_ptr() - flat.data_ptr()) % 16 == 0
    flat, view = guarded((7,), "f32", "cpu")
    assert view.is_contiguous() and (view.data_ptr() - flat.data_ptr()) % 16 == 0
