"""The benchmark's host-side bookkeeping, on CPU: the source hash that keys the
recorded ncu traffic ignores comments and blank space but not code (a kernel
whose code changed reports its traffic as null until it is measured again)."""
import bench


def test_code_only_ignores_comments_and_spacing():
    a = "int f(int x) {  // doubles\n  return 2 * x;   /* block\ncomment */\n}\n"
    b = "int f(int x) {\n\n    return 2 * x;\n}   // other words\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_sees_code_changes():
    a = "int f(int x) { return 2 * x; }  // same comment\n"
    b = "int f(int x) { return 3 * x; }  // same comment\n"
    assert bench._code_only(a) != bench._code_only(b)

